"""GPU parity of the randomised gate options (noisy_gate_policy = rsample /
jitter, second-expert sampling, random token selection), all drawn inside
the layer from Philox4x32-10 keyed by (seed, offset):
  * the draws: uniforms and queue positions bit for bit against the
    oracle's own Philox; the Gumbel noise within float32 rounding;
  * routing bit-exact against the oracle fed the GPU's fp32 logits and the
    GPU's Gumbel noise (the selection keys are float32 sums on both sides);
  * y end to end and, under jitter, the gradients, against the oracle."""
import numpy as np
import pytest
import torch

from _harness import (DEV, GpuRun, WORKLOADS, assert_close, check_routing_equal, f64, i64,
                      oracle_cfg)
from mixture_experts_layer_86_b300 import _native as N
from mixture_experts_layer_86_b300.inputs import Workload
from oracle import moe_oracle as O
from oracle import random_streams as RS

pytestmark = pytest.mark.gpu

SEED, OFFSET = (0x1234 << 32) | 0x5678, (3 << 32) | 11


def _wl(base, S, **kw):
    b = WORKLOADS[base]
    return Workload(f"{base}_noise", S, b.hidden_size if base != "e8_bf16" else 512,
                    b.ffn_size if base != "e8_bf16" else 256, b.num_experts, b.k,
                    kw.pop("cf", b.capacity_factor), b.min_capacity, b.drop_tokens, b.act, b.dtype,
                    seed=b.seed, bias_std=0.1, noise_seed=SEED, noise_offset=OFFSET, **kw)


def _ocfg(wl):
    c = oracle_cfg(wl)
    c.noise_policy, c.second_expert_sampling, c.use_rts = (
        wl.noise_policy, wl.second_expert_sampling, wl.use_rts)
    c.noise_seed, c.noise_offset, c.jitter_eps = wl.noise_seed, wl.noise_offset, wl.jitter_eps
    c.dtype = wl.dtype
    return c


def _gpu_noise(cfg, S, E):
    u = torch.empty((S, E), dtype=torch.float32, device=DEV)
    g = torch.empty_like(u)
    pos = torch.empty((S,), dtype=torch.int32, device=DEV)
    N.moe_gate_noise(cfg, u, g, pos)
    torch.cuda.synchronize()
    return u, g, pos


@pytest.mark.parametrize("S,E", [(1, 2), (1000, 8), (4097, 64), (16384, 256)])
def test_gate_draws_match_the_oracle(S, E):
    cfg = N.make_config(S, 64, 64, E, 2, 1.0, 4, True, noise_seed=SEED, noise_offset=OFFSET)
    u, g, pos = _gpu_noise(cfg, S, E)
    ou, og = RS.gate_noise(S, E, SEED, OFFSET)
    assert np.array_equal(f64(u), ou)                        # Philox words, bit for bit
    assert np.allclose(f64(g), og, rtol=2e-6, atol=2e-6)     # -ln(-ln u), float32 logf
    assert np.array_equal(i64(pos), RS.rts_position(S, SEED, OFFSET))
    # another offset is another draw
    cfg2 = N.make_config(S, 64, 64, E, 2, 1.0, 4, True, noise_seed=SEED, noise_offset=OFFSET + 1)
    u2, _, _ = _gpu_noise(cfg2, S, E)
    if S > 1:
        assert not torch.equal(u, u2)


CASES = [
    ("e8_bf16", 1500, dict(noise_policy="rsample")),
    ("e8_bf16", 1500, dict(second_expert_sampling=True)),
    ("e8_bf16", 1500, dict(use_rts=True, cf=0.6)),
    ("e8_bf16", 1500, dict(noise_policy="jitter", jitter_eps=0.05)),
    ("e8_bf16", 1500, dict(noise_policy="rsample", use_rts=True, cf=0.6)),
    ("tiny_fp32", 256, dict(noise_policy="rsample", use_rts=True)),
    ("tiny_fp32", 256, dict(noise_policy="jitter", jitter_eps=0.1)),
    ("e64_bf16", 300, dict(second_expert_sampling=True, use_rts=True, cf=0.8)),
]


@pytest.mark.parametrize("base,S,kw", CASES, ids=lambda c: str(c))
def test_noisy_forward_parity(base, S, kw):
    wl = _wl(base, S, **kw)
    run = GpuRun(wl, training=True)
    c = _ocfg(wl)
    _, g_gpu, _ = _gpu_noise(run.cfg, S, wl.num_experts)
    # routing: the oracle on the GPU's fp32 logits and the GPU's noise
    ref_rt = O.route(f64(run.bufs["logits"]), c, noise=f64(g_gpu))
    check_routing_equal(run, ref_rt)
    assert np.allclose(f64(run.bufs["topk_w"]), ref_rt["weights"], rtol=2e-6, atol=1e-7)
    assert abs(float(run.l_aux.item()) - ref_rt["l_aux"]) <= 1e-5 * abs(ref_rt["l_aux"])
    inp = run.inp
    # the logits: the oracle's own (jitter included) in float64
    lb = None if inp.logit_bias is None else f64(inp.logit_bias)
    own = O.gate_logits(O.router_input(f64(inp.x), c)[0], f64(inp.w_gate), lb)
    got = f64(run.bufs["logits"])
    assert np.abs(got - own).max() <= 1e-5 * np.abs(own).max()
    # y under the GPU's routing
    assert_close(f64(run.y), _y_under(run, c, ref_rt), wl.dtype, "y")
    assert N.moe_get_device_error() == 0


def _y_under(run, c, g):
    """The oracle's y under routing g (the GPU's), from the inputs."""
    inp = run.inp
    rt = g["routing"]
    x_disp = O.dispatch(f64(inp.x), rt)
    _, _, out = O.expert_ffn(x_disp, rt.offsets, f64(inp.w1), f64(inp.b1), f64(inp.w2),
                             f64(inp.b2), c.act)
    return O.combine(out, rt, g["weights"], run.wl.hidden_size)


def test_rts_changes_which_tokens_are_dropped():
    wl = _wl("e8_bf16", 2000, cf=0.4)
    plain = GpuRun(wl)
    rts = GpuRun(_wl("e8_bf16", 2000, cf=0.4, use_rts=True))
    assert torch.equal(plain.bufs["topk_idx"], rts.bufs["topk_idx"])
    assert torch.equal(plain.kept, rts.kept)
    kept_plain = plain.bufs["slot"] >= 0
    kept_rts = rts.bufs["slot"] >= 0
    assert kept_plain.sum() == kept_rts.sum()
    assert not torch.equal(kept_plain, kept_rts)
    # in token order the dropped first choices pile up at the end of the batch
    S = wl.num_tokens
    late = lambda kept: float((~kept[S // 2:, 0]).sum()) / max(1.0, float((~kept[:, 0]).sum()))
    assert late(kept_plain) > 0.9 and late(kept_rts) < 0.75


@pytest.mark.parametrize("kw", [dict(noise_policy="jitter", jitter_eps=0.05),
                                dict(noise_policy="rsample", use_rts=True, cf=0.6)])
def test_noisy_backward_parity(kw):
    wl = _wl("train_e32", 900, **kw)
    wl = Workload(wl.name, wl.num_tokens, wl.hidden_size, wl.ffn_size, wl.num_experts, wl.k,
                  wl.capacity_factor, wl.min_capacity, wl.drop_tokens, wl.act, wl.dtype,
                  seed=wl.seed, bias_std=0.1, aux_loss_weight=0.01, backward=True,
                  noise_policy=wl.noise_policy, second_expert_sampling=wl.second_expert_sampling,
                  use_rts=wl.use_rts, jitter_eps=wl.jitter_eps, noise_seed=SEED,
                  noise_offset=OFFSET)
    run = GpuRun(wl, training=True)
    run.backward()
    c = _ocfg(wl)
    _, g_gpu, _ = _gpu_noise(run.cfg, wl.num_tokens, wl.num_experts)
    inp = run.inp
    ref_rt = O.route(f64(run.bufs["logits"]), c, noise=f64(g_gpu))
    check_routing_equal(run, ref_rt)
    ref = O.forward(c, f64(inp.x), f64(inp.w_gate), f64(inp.w1), f64(inp.b1), f64(inp.w2),
                    f64(inp.b2), logit_bias=None if inp.logit_bias is None else f64(inp.logit_bias),
                    logits=f64(run.bufs["logits"]))
    # the forward above re-routes with the oracle's own noise; use the GPU's
    ref.update(ref_rt)
    rt = ref_rt["routing"]
    ref["x_disp"] = O.dispatch(f64(inp.x), rt)
    ref["h_pre"], ref["h"], ref["out"] = O.expert_ffn(ref["x_disp"], rt.offsets, f64(inp.w1),
                                                      f64(inp.b1), f64(inp.w2), f64(inp.b2), c.act)
    gref = O.backward(c, ref, f64(inp.x), f64(inp.w_gate), f64(inp.w1), f64(inp.w2), f64(inp.dy))
    for key in ("dx", "dw_gate", "dw1", "db1", "dw2", "db2"):
        assert_close(f64(run.grads[key]), gref[key], wl.dtype, key)
    assert N.moe_get_device_error() == 0
