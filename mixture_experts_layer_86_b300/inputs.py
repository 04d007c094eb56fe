"""Seeded synthetic inputs for the MoE layer workloads.

This module only draws random tensors and names the workload shapes; it holds
none of the layer's arithmetic, so that the CUDA path and the float64 oracle
can be fed identical inputs without sharing code.

Recipe (every workload): a CPU ``torch.Generator`` seeded with the workload's
seed draws, in this order and in float32,
  x ~ N(0,1)                    [S, d]
  W_g ~ N(0, 1/d)               [E, d]        (nn.Linear layout: out x in)
  W1 ~ N(0, 1/d)                [E, f, d]     (fan_in = d)
  W2 ~ N(0, 1/f)                [E, d, f]     (fan_in = f)
  b1 ~ N(0, bias_std^2)         [E, f]        (zero when bias_std == 0)
  b2 ~ N(0, bias_std^2)         [E, d]
  dY ~ N(0,1)                   [S, d]        (only when a backward is run)
and casts each to the workload dtype with round-to-nearest-even.  The
skewed-routing workload adds a constant per-expert logit bias
b_e = skew * ln(1/(e+1)) (fp32), i.e. expert e has Zipf rank e.  A workload
with gate noise finally draws a per-token logit noise [S, E] ~
N(0, logit_noise_std^2) (fp32); the logit bias is then [S, E].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Dict, Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    num_tokens: int
    hidden_size: int
    ffn_size: int
    num_experts: int
    k: int
    capacity_factor: float
    min_capacity: int
    drop_tokens: bool
    act: str              # "relu" | "gelu_tanh" | "gelu_erf"
    dtype: str            # "f32" | "bf16"
    seed: int
    skew: float = 0.0     # per-expert logit bias coefficient (0 = none)
    bias_std: float = 0.0
    aux_loss_weight: float = 0.0
    backward: bool = False
    gate_temperature: float = 1.0   # softmax temperature of the gate
    aux_loss_type: str = "load"     # "load" | "std"
    logit_noise_std: float = 0.0    # > 0: per-token gate noise N(0, std^2), [S, E]
    noise_policy: str = "none"      # in-layer gate noise: "none" | "jitter" | "rsample"
    second_expert_sampling: bool = False
    use_rts: bool = False           # random token selection
    jitter_eps: float = 0.01
    noise_seed: int = 0
    noise_offset: int = 0

    def scaled(self, num_tokens: int, **kw) -> "Workload":
        """Same layer shape and routing settings with a different batch."""
        return replace(self, num_tokens=num_tokens,
                       name=f"{self.name}@S{num_tokens}", **kw)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


# The five layer configurations the implementation is specified and measured
# on, and the inference (decode) shape of the 64-expert layer.
WORKLOADS: Dict[str, Workload] = {
    # tiny fp32 forward, ReLU, k=1
    "tiny_fp32": Workload("tiny_fp32", 256, 32, 64, 4, 1, 1.0, 4, True,
                          "relu", "f32", seed=0),
    # bf16 forward, 8 experts, top-2
    "e8_bf16": Workload("e8_bf16", 4096, 512, 2048, 8, 2, 1.0, 4, True,
                        "gelu_tanh", "bf16", seed=1),
    # fine-grained bf16 forward, 64 experts (DeepSeek-MoE sized experts)
    "e64_bf16": Workload("e64_bf16", 16384, 2048, 5120, 64, 2, 1.25, 4, True,
                         "gelu_tanh", "bf16", seed=2),
    # skewed routing, with and without the capacity cap
    "skew_e16_drop": Workload("skew_e16_drop", 8192, 1024, 4096, 16, 2, 2.0, 4,
                              True, "gelu_tanh", "bf16", seed=3, skew=1.2),
    "skew_e16_nodrop": Workload("skew_e16_nodrop", 8192, 1024, 4096, 16, 2, 2.0,
                                4, False, "gelu_tanh", "bf16", seed=3, skew=1.2),
    # training step: forward + backward with l_aux weight 0.01
    "train_e32": Workload("train_e32", 8192, 1024, 4096, 32, 2, 1.25, 4, True,
                          "gelu_tanh", "bf16", seed=4, aux_loss_weight=0.01,
                          backward=True),
    # inference: one decode step of 256 sequences through the 64-expert
    # layer, with the evaluation capacity factor (1.0) as the capacity
    # factor; every expert sees a handful of tokens, so the expert GEMMs
    # stream the weights and are bound by HBM, not by the tensor cores
    "decode_e64": Workload("decode_e64", 256, 2048, 5120, 64, 2, 1.0, 4, True,
                           "gelu_tanh", "bf16", seed=5),
}


@dataclass
class LayerInputs:
    x: torch.Tensor
    w_gate: torch.Tensor
    w1: torch.Tensor
    b1: torch.Tensor
    w2: torch.Tensor
    b2: torch.Tensor
    logit_bias: Optional[torch.Tensor]
    dy: Optional[torch.Tensor]

    def to(self, device) -> "LayerInputs":
        mv = lambda t: None if t is None else t.to(device)  # noqa: E731
        return LayerInputs(*(mv(getattr(self, f)) for f in
                             ("x", "w_gate", "w1", "b1", "w2", "b2",
                              "logit_bias", "dy")))


def make_inputs(wl: Workload, with_dy: Optional[bool] = None,
                seed: Optional[int] = None) -> LayerInputs:
    """Draw the workload's tensors on the CPU (see the module docstring)."""
    g = torch.Generator().manual_seed(wl.seed if seed is None else seed)
    S, d, f, E = wl.num_tokens, wl.hidden_size, wl.ffn_size, wl.num_experts
    dt = wl.torch_dtype

    def draw(shape, std):
        return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(dt)

    x = draw((S, d), 1.0)
    w_gate = draw((E, d), 1.0 / math.sqrt(d))
    w1 = draw((E, f, d), 1.0 / math.sqrt(d))
    w2 = draw((E, d, f), 1.0 / math.sqrt(f))
    if wl.bias_std > 0:
        b1 = draw((E, f), wl.bias_std)
        b2 = draw((E, d), wl.bias_std)
    else:
        b1 = torch.zeros((E, f), dtype=dt)
        b2 = torch.zeros((E, d), dtype=dt)
    dy = None
    if wl.backward if with_dy is None else with_dy:
        dy = draw((S, d), 1.0)
    logit_bias = skew_logit_bias(wl)
    if wl.logit_noise_std > 0:
        # noisy gating: the caller's per-token logit noise, drawn last so the
        # other tensors do not depend on it
        noise = torch.randn((S, E), generator=g, dtype=torch.float32) * wl.logit_noise_std
        logit_bias = noise if logit_bias is None else noise + logit_bias[None, :]
    return LayerInputs(x, w_gate, w1, b1, w2, b2, logit_bias, dy)


def skew_logit_bias(wl: Workload) -> Optional[torch.Tensor]:
    """The skewed workload's per-expert logit bias b_e = skew * ln(1/(e+1))
    (fp32), or None when the workload has no skew."""
    if not wl.skew:
        return None
    return torch.tensor([wl.skew * math.log(1.0 / (e + 1)) for e in range(wl.num_experts)],
                        dtype=torch.float32)


def make_residual_weights(wl: Workload):
    """Weights of PR-MoE's residual MLP for a workload, drawn like one
    expert's: a CPU generator seeded with seed + 1000 draws, in float32,
    rw1 ~ N(0, 1/d) [f, d], rw2 ~ N(0, 1/f) [d, f], then rb1 [f] and rb2 [d]
    ~ N(0, bias_std^2) (zero when bias_std == 0), cast to the layer dtype."""
    g = torch.Generator().manual_seed(wl.seed + 1000)
    d, f, dt = wl.hidden_size, wl.ffn_size, wl.torch_dtype

    def draw(shape, std):
        return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(dt)

    rw1 = draw((f, d), 1.0 / math.sqrt(d))
    rw2 = draw((d, f), 1.0 / math.sqrt(f))
    if wl.bias_std > 0:
        rb1, rb2 = draw((f,), wl.bias_std), draw((d,), wl.bias_std)
    else:
        rb1, rb2 = torch.zeros((f,), dtype=dt), torch.zeros((d,), dtype=dt)
    return rw1, rb1, rw2, rb2


def make_residual_mix(wl: Workload):
    """Weights of PR-MoE's learned two-way mix for a workload: a CPU
    generator seeded with seed + 2000 draws, in float32, mix_w ~ N(0, 1/d)
    [2, d] then mix_b ~ N(0, 0.5^2) [2], cast to the layer dtype."""
    g = torch.Generator().manual_seed(wl.seed + 2000)
    d, dt = wl.hidden_size, wl.torch_dtype
    mix_w = (torch.randn((2, d), generator=g, dtype=torch.float32) / math.sqrt(d)).to(dt)
    mix_b = (torch.randn((2,), generator=g, dtype=torch.float32) * 0.5).to(dt)
    return mix_w, mix_b


def make_gate_inputs(wl: Workload):
    """x, W_g and the logit bias exactly as make_inputs draws them (the first
    two draws of the recipe), without drawing the expert weights."""
    g = torch.Generator().manual_seed(wl.seed)
    S, d, E = wl.num_tokens, wl.hidden_size, wl.num_experts

    def draw(shape, std):
        return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(wl.torch_dtype)

    x = draw((S, d), 1.0)
    w_gate = draw((E, d), 1.0 / math.sqrt(d))
    return x, w_gate, skew_logit_bias(wl)
