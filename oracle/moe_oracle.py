"""Float64 CPU oracle of the top-k gated Mixture-of-Experts FFN layer.

TEST INFRASTRUCTURE ONLY.  This module is imported by ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py``; the product path never imports it.  It shares no code
with the CUDA library: it is written from the pages' description of the
layer, step by step, in the plainest form (NumPy float64, sequential loops
where the definition is sequential).

Sources (web pages on the MoE layer; cited by address and section):

* [deepspeed.moe overview]  adg.csdn.net/694deb285b9f5f31781ae763 --
  §2.1 "MoE 层" (constructor arguments ``hidden_size, num_experts, k,
  capacity_factor, min_capacity, drop_tokens``; return value
  ``(output, gate_loss, expert_count)``) and §3.1 "MoE 层前向传播"
  (gate -> top-k -> dispatch -> experts -> weighted combine -> balance loss).
* [DeepSeek-MoE traps]  lnwmold.com/news/1162317 -- ch.1 ``moe_forward``
  pseudocode (softmax, top-2, ``output += expert_out * top_weights``),
  ch.1 load-balancing table (capacity = ceil(seq_len*2/num_experts*cf)),
  §3.1 ``TopKRouter`` (gradient reaches only the selected logits),
  §2.1/§2.3 (experts that receive no token get a zero gradient).
* [MoE explainer]  lpnh.cn/news/725941 -- §3.1 ``MoELayer`` pseudocode:
  Step 1 router logits, Step 2 top-k then softmax over the k selected
  logits, Step 3 flatten & scatter, Step 4 expert FFN
  (Linear -> GELU -> Linear), Step 5 gather weighted sum; capacity and
  drop-tokens comments.
* [ZeRO-3 + MoE in practice]  mhpq.cn/news/1113018 -- §3.2 worked capacity
  arithmetic; §2.2 drop / overflow discussion.

Readings where the pages are silent or disagree:

R1  Top-k is taken on the logits (softmax is monotone, so the selected set is
    the same); ties go to the LOWER expert index.
R2  k=2 weights are renormalised over the two selected experts
    (softmax over the two selected logits == p_i / (p_1 + p_2)); k=1 uses the
    raw softmax probability (``output += expert_out * top_weights`` with no
    renormalisation).  Renormalisation happens before any token is dropped.
R3  capacity C = max(min_capacity, ceil(S*k*cf/E)), cf read as an exact
    decimal; ``drop_tokens=False`` means no cap at all.
R4  Slots are handed out in priority order: every first choice, in token
    order, before any second choice.  A slot >= C is dropped.
R5  l_aux = E * sum_e mean_s(p[s,e]) * first[e]/S, first[e] counting first
    choices before dropping.
R6  A token whose every slot is dropped contributes y_s = 0 (no residual).
R7  "GeLU" without qualifier is the tanh form.
R8  PR-MoE's residual expert (use_residual=True) is combined with the MoE
    output by a sum, y = MoE(x) + MLP(x); the page gives no mixing formula.
    The other reading offered: a learned per-token two-way mix,
    c = softmax(x W_c^T + b_c) over 2 entries, y = c0 MoE(x) + c1 MLP(x).
R9  The std-based balance loss lambda * (std(usage_prob) + 1e-6) reads
    usage_prob[e] as mean_s p[s,e] (the differentiable usage), with the
    population std over experts.
R10 The gate temperature T (gating_softmax_temp) divides the logits before
    the softmax; the top-k choice (taken on the logits) is unchanged.
    Noisy gating adds caller-drawn noise to the logits as a per-token bias
    [S,E] (the layer itself stays deterministic; the noise gets no gradient).
R11 In-layer randomness (``noisy_gate_policy``, ``use_rts``,
    ``top2_2nd_expert_sampling``, named on the deepspeed.moe overview §2.1
    without formulas) comes from Philox4x32-10 keyed by a seed and an offset
    (``random_streams``).  noisy_gate_policy = "rsample": the experts are
    chosen as the top-k of logits + g, g[s,e] standard Gumbel noise (the
    Gumbel-max sample of the softmax); the keys are formed in float32, the
    precision of the logits; probabilities and combine weights stay those of
    the noise-free logits.  The noise is a constant of the backward.
R12 noisy_gate_policy = "jitter": the router sees x~ = x * f, f[s,c] =
    1 + eps * (2u - 1) (eps = 0.01 unless configured), computed in float32
    and, for a bf16 layer, rounded to bf16; the experts see x.  Backward:
    dW_g = dlogits^T x~ and the router's part of dX is (dlogits W_g) * f.
R13 top2_2nd_expert_sampling: the first choice is the noise-free arg-max;
    the second is the arg-max of the float32 keys logits + g over the other
    experts.
R14 use_rts (random token selection): the capacity queue takes every first
    choice before every second choice, as in R4, but within a choice level
    the tokens come in the order of a keyed pseudorandom permutation pi
    (a Feistel network over Philox, cycle-walked to [0, S)) instead of token
    order; rows of the expert-major buffer follow the queue.

Parity pins (tests/test_oracle_pins.py): brute-force top-k and slot
enumeration on tiny inputs, hand-worked capacity/drop cases, the pages' own
capacity arithmetic, closed-form l_aux cases, dense equivalence with
``drop_tokens=False``, E=1 identity, and central finite differences of the
backward pass.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from fractions import Fraction
from typing import Optional

import numpy as np

from . import random_streams as RS

ACT_RELU = "relu"
ACT_GELU_TANH = "gelu_tanh"
ACT_GELU_ERF = "gelu_erf"

_SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)


# ---------------------------------------------------------------------------
# capacity  ([DeepSeek-MoE traps] ch.1 load-balancing table; [MoE explainer]
# §3.1 expert_capacity comment; [deepspeed.moe overview] §2.1 min_capacity,
# drop_tokens)
# ---------------------------------------------------------------------------
def capacity(num_tokens: int, num_experts: int, k: int, capacity_factor,
             min_capacity: int, drop_tokens: bool) -> Optional[int]:
    """Per-expert token capacity, exact; ``None`` means unbounded.

    C = max(min_capacity, ceil(S * k * cf / E)) with cf taken as the decimal
    it is written as (``Fraction(str(cf))``), so 1.25 and 1.2 are exact.
    """
    if not drop_tokens:
        return None
    cf = Fraction(str(capacity_factor))
    raw = Fraction(num_tokens * k) * cf / num_experts
    return max(int(min_capacity), math.ceil(raw))


# ---------------------------------------------------------------------------
# gate: logits, softmax, top-k, weights, aux loss
# ---------------------------------------------------------------------------
def gate_logits(x: np.ndarray, w_gate: np.ndarray,
                logit_bias: Optional[np.ndarray] = None) -> np.ndarray:
    """Router logits [S,E] = x @ W_g^T (+ b) in float64.

    [MoE explainer] §3.1 Step 1 (``router = nn.Linear(hidden, E)``);
    [DeepSeek-MoE traps] ch.1 ``logits = router(x)``.
    """
    lg = np.asarray(x, np.float64) @ np.asarray(w_gate, np.float64).T
    if logit_bias is not None:
        b = np.asarray(logit_bias, np.float64)
        lg = lg + (b[None, :] if b.ndim == 1 else b)   # [E] or per-token [S,E]
    return lg


def softmax(logits: np.ndarray) -> np.ndarray:
    """Row softmax over experts, float64 ([DeepSeek-MoE traps] ch.1)."""
    lg = np.asarray(logits, np.float64)
    z = np.exp(lg - lg.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def topk_experts(logits: np.ndarray, k: int) -> np.ndarray:
    """idx[S,k]: choice 1 is the arg-max logit, choice 2 the arg-max of the
    rest; equal logits go to the lower index (reading R1).

    ``np.argmax`` returns the first (lowest) index of the maximum, which is
    exactly the tie-break rule.
    """
    lg = np.array(logits, np.float64, copy=True)
    S, E = lg.shape
    if not 1 <= k <= E:
        raise ValueError("k must be in [1, E]")
    idx = np.empty((S, k), np.int64)
    rows = np.arange(S)
    for j in range(k):
        c = np.argmax(lg, axis=1)
        idx[:, j] = c
        lg[rows, c] = -np.inf
    return idx


def gate_weights(probs: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Combine weights w[S,k] (reading R2).

    k=2: softmax over the two selected logits, i.e. p_j / (p_1 + p_2)
    ([MoE explainer] §3.1 Step 2).  k=1: the raw probability p_1
    ([DeepSeek-MoE traps] ch.1 ``output += expert_out * top_weights``).
    """
    p_sel = np.take_along_axis(np.asarray(probs, np.float64), idx, axis=1)
    if idx.shape[1] == 1:
        return p_sel
    return p_sel / p_sel.sum(axis=1, keepdims=True)


def aux_loss(probs: np.ndarray, idx: np.ndarray, kind: str = "load") -> float:
    """Load-balancing loss.

    ``load``: l_aux = E * sum_e mean_s(p[s,e]) * first[e]/S.  The pages name
    the term (``gate_loss``, weight 0.01) without a formula; this is the
    definition the layer is specified with (reading R5).
    ``std``: the DeepSeek-MoE page's alternative, lambda * (std(usage_prob)
    + 1e-6) ([DeepSeek-MoE traps] ch.1 load-balancing table); reading R9:
    usage_prob[e] = mean_s p[s,e], std over experts (population).
    """
    p = np.asarray(probs, np.float64)
    S, E = p.shape
    if kind == "std":
        u = p.mean(axis=0)
        return float(np.sqrt(np.mean((u - u.mean()) ** 2)) + 1e-6)
    first = np.bincount(idx[:, 0], minlength=E).astype(np.float64)
    return float(E * np.sum(p.mean(axis=0) * (first / S)))


# ---------------------------------------------------------------------------
# slot assignment, drop mask and counts
# ---------------------------------------------------------------------------
@dataclass
class Routing:
    idx: np.ndarray        # [S,k] int64 expert of each choice
    slot: np.ndarray       # [S,k] int64 position in the expert's queue, -1 = dropped
    routed: np.ndarray     # [E] int64 tokens that chose the expert (before drop)
    kept: np.ndarray       # [E] int64 tokens kept (<= capacity)
    offsets: np.ndarray    # [E+1] int64 exclusive scan of kept
    row_src: np.ndarray    # [R] int64 row r of the expert-major buffer holds choice s*k+j
    capacity: Optional[int]

    @property
    def num_rows(self) -> int:
        return int(self.offsets[-1])

    def row_of(self, s: int, j: int) -> int:
        """Row in the expert-major buffer of (token s, choice j), -1 if dropped."""
        sl = int(self.slot[s, j])
        if sl < 0:
            return -1
        return int(self.offsets[self.idx[s, j]]) + sl


def assign_slots(idx: np.ndarray, num_experts: int,
                 cap: Optional[int], order=None) -> Routing:
    """Capacity-limited slot assignment in priority order (reading R4).

    One counter per expert; walk choice j = 0..k-1 (outer) and token
    s = 0..S-1 (inner); the current counter value is the slot and the
    counter advances whether or not the slot is kept.  Kept iff slot < C
    ([deepspeed.moe overview] §2.1 drop_tokens; [MoE explainer] §3.1 "Drop
    tokens").  Rows of the expert-major buffer are offsets[e] + slot.
    ``order``: the tokens in queue order within a choice level (random token
    selection, reading R14); token order when None.
    """
    S, k = idx.shape
    counter = [0] * num_experts
    slot = np.full((S, k), -1, np.int64)
    tokens = range(S) if order is None else [int(t) for t in order]
    for j in range(k):
        for s in tokens:
            e = int(idx[s, j])
            pos = counter[e]
            counter[e] += 1
            if cap is None or pos < cap:
                slot[s, j] = pos
    routed = np.array(counter, np.int64)
    kept = routed.copy() if cap is None else np.minimum(routed, cap)
    offsets = np.zeros(num_experts + 1, np.int64)
    offsets[1:] = np.cumsum(kept)
    row_src = np.full(int(offsets[-1]), -1, np.int64)
    for s in range(S):
        for j in range(k):
            if slot[s, j] >= 0:
                row_src[offsets[idx[s, j]] + slot[s, j]] = s * k + j
    return Routing(idx=idx, slot=slot, routed=routed, kept=kept,
                   offsets=offsets, row_src=row_src, capacity=cap)


# ---------------------------------------------------------------------------
# dispatch, expert FFN, combine
# ---------------------------------------------------------------------------
def dispatch(x: np.ndarray, rt: Routing) -> np.ndarray:
    """Expert-major copy of the kept token rows ([MoE explainer] §3.1 Step 3
    "flatten & scatter"): row offsets[e]+slot holds x[s]."""
    x = np.asarray(x, np.float64)
    out = np.zeros((rt.num_rows, x.shape[1]), np.float64)
    S, k = rt.idx.shape
    for s in range(S):
        for j in range(k):
            r = rt.row_of(s, j)
            if r >= 0:
                out[r] = x[s]
    return out


def activation(z: np.ndarray, act: str) -> np.ndarray:
    """ReLU, tanh-GeLU or erf-GeLU ([MoE explainer] §3.1 Step 4: GELU)."""
    z = np.asarray(z, np.float64)
    if act == ACT_RELU:
        return np.maximum(z, 0.0)
    if act == ACT_GELU_TANH:
        return 0.5 * z * (1.0 + np.tanh(_SQRT_2_OVER_PI * (z + 0.044715 * z ** 3)))
    if act == ACT_GELU_ERF:
        from scipy.special import erf
        return 0.5 * z * (1.0 + erf(z / math.sqrt(2.0)))
    raise ValueError(act)


def activation_grad(z: np.ndarray, act: str) -> np.ndarray:
    """d act / d z, analytically."""
    z = np.asarray(z, np.float64)
    if act == ACT_RELU:
        return (z > 0.0).astype(np.float64)
    if act == ACT_GELU_TANH:
        u = _SQRT_2_OVER_PI * (z + 0.044715 * z ** 3)
        t = np.tanh(u)
        du = _SQRT_2_OVER_PI * (1.0 + 3.0 * 0.044715 * z ** 2)
        return 0.5 * (1.0 + t) + 0.5 * z * (1.0 - t * t) * du
    if act == ACT_GELU_ERF:
        from scipy.special import erf
        pdf = np.exp(-0.5 * z * z) / math.sqrt(2.0 * math.pi)
        return 0.5 * (1.0 + erf(z / math.sqrt(2.0))) + z * pdf
    raise ValueError(act)


def expert_ffn(x_disp: np.ndarray, offsets: np.ndarray, w1: np.ndarray,
               b1: np.ndarray, w2: np.ndarray, b2: np.ndarray, act: str):
    """Per-expert FFN on its contiguous rows ([MoE explainer] §3.1 Step 4):
    h_pre = x W1_e^T + b1_e, h = act(h_pre), out = h W2_e^T + b2_e.

    Weights in nn.Linear layout: w1[E,f,d], w2[E,d,f].  Returns
    (h_pre, h, out) in float64.
    """
    E = w1.shape[0]
    R = x_disp.shape[0]
    f, d = w1.shape[1], w1.shape[2]
    h_pre = np.zeros((R, f), np.float64)
    out = np.zeros((R, d), np.float64)
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a == b:
            continue
        h_pre[a:b] = x_disp[a:b] @ np.asarray(w1[e], np.float64).T + np.asarray(b1[e], np.float64)
        he = activation(h_pre[a:b], act)
        out[a:b] = he @ np.asarray(w2[e], np.float64).T + np.asarray(b2[e], np.float64)
    return h_pre, activation(h_pre, act), out


def combine(out_disp: np.ndarray, rt: Routing, w: np.ndarray, d: int) -> np.ndarray:
    """y_s = sum over kept choices j of w[s,j] * out[row(s,j)]
    ([MoE explainer] §3.1 Step 5; [deepspeed.moe overview] §3.1 item 4
    weighted merge).  A token with no kept choice gets 0 (reading R6)."""
    S, k = rt.idx.shape
    y = np.zeros((S, d), np.float64)
    for s in range(S):
        for j in range(k):
            r = rt.row_of(s, j)
            if r >= 0:
                y[s] += w[s, j] * out_disp[r]
    return y


# ---------------------------------------------------------------------------
# whole layer
# ---------------------------------------------------------------------------
@dataclass
class LayerConfig:
    num_tokens: int
    hidden_size: int
    ffn_size: int
    num_experts: int
    k: int
    capacity_factor: float
    min_capacity: int
    drop_tokens: bool
    act: str
    aux_loss_weight: float = 0.0
    gate_temperature: float = 1.0   # p = softmax(logits / T) (reading R10)
    aux_loss_type: str = "load"     # "load" | "std"
    noise_policy: str = "none"      # "none" | "jitter" | "rsample" (R11, R12)
    second_expert_sampling: bool = False   # R13
    use_rts: bool = False           # R14
    noise_seed: int = 0
    noise_offset: int = 0
    jitter_eps: float = 0.01
    dtype: str = "bf16"             # the router input's storage under jitter: bf16 | f32 | f64


def uses_selection_noise(cfg: LayerConfig) -> bool:
    """Whether the expert choice reads Gumbel keys (R11 rsample, R13
    second-expert sampling with k = 2)."""
    return cfg.noise_policy == "rsample" or (cfg.second_expert_sampling and cfg.k == 2)


def selection_noise(cfg: LayerConfig, num_tokens: int) -> Optional[np.ndarray]:
    """The Gumbel noise g[s,e] the choice uses (R11, R13), or None."""
    if uses_selection_noise(cfg):
        return RS.gate_noise(num_tokens, cfg.num_experts, cfg.noise_seed, cfg.noise_offset)[1]
    return None


def select_experts(logits: np.ndarray, cfg: LayerConfig, noise=None) -> np.ndarray:
    """The k chosen experts per token under the gate-noise options: plain
    top-k of the logits; top-k of the float32 keys logits + g (rsample,
    R11); or the noise-free first choice and the second from the keys
    (second-expert sampling, R13).  ``noise``: g (float, [S,E]); drawn from
    the layer's stream when None; ignored when neither option is on (jitter
    and random token selection leave the choice on the logits)."""
    lg = np.asarray(logits, np.float64)
    S = lg.shape[0]
    if not uses_selection_noise(cfg):
        return topk_experts(lg, cfg.k)
    if noise is None:
        noise = selection_noise(cfg, S)
    keys = (lg.astype(np.float32) + np.asarray(noise).astype(np.float32)).astype(np.float64)
    if cfg.noise_policy == "rsample":
        return topk_experts(keys, cfg.k)
    first = topk_experts(lg, 1)[:, 0]
    rest = keys.copy()
    rest[np.arange(S), first] = -np.inf
    second = np.argmax(rest, axis=1)        # ties to the lower index
    return np.stack([first, second], axis=1)


def router_input(x: np.ndarray, cfg: LayerConfig):
    """(x~, f): the router's input and the jitter factors (R12); (x, None)
    without jitter."""
    x = np.asarray(x, np.float64)
    if cfg.noise_policy != "jitter":
        return x, None
    S, d = x.shape
    f = RS.jitter_factors(S, d, cfg.jitter_eps, cfg.noise_seed, cfg.noise_offset)
    if cfg.dtype == "f64":
        return x * f.astype(np.float64), f
    prod = x.astype(np.float32) * f                     # one float32 rounding
    if cfg.dtype == "bf16":
        import torch
        prod = torch.from_numpy(prod).to(torch.bfloat16).to(torch.float32).numpy()
    return prod.astype(np.float64), f


def route(logits: np.ndarray, cfg: LayerConfig, noise=None) -> dict:
    """Gate stages after the logits: softmax, top-k, weights, slots, l_aux."""
    S, E = logits.shape
    probs = softmax(np.asarray(logits, np.float64) / cfg.gate_temperature)
    idx = select_experts(logits, cfg, noise)
    w = gate_weights(probs, idx)
    cap = capacity(S, E, cfg.k, cfg.capacity_factor, cfg.min_capacity,
                   cfg.drop_tokens)
    order = None
    if cfg.use_rts:
        order = np.argsort(RS.rts_position(S, cfg.noise_seed, cfg.noise_offset), kind="stable")
    rt = assign_slots(idx, E, cap, order)
    return {"logits": np.asarray(logits, np.float64), "probs": probs,
            "weights": w, "routing": rt, "l_aux": aux_loss(probs, idx, cfg.aux_loss_type)}


def forward(cfg: LayerConfig, x, w_gate, w1, b1, w2, b2, logit_bias=None,
            logits: Optional[np.ndarray] = None) -> dict:
    """The whole layer; returns every intermediate in float64.

    ``logits`` overrides the oracle's own gate GEMM (used to route on the
    exact fp32 logits another implementation produced).  Returns
    ``y``, ``l_aux``, ``routing`` (with ``kept`` = expert_count), ``weights``,
    ``probs``, ``x_disp``, ``h_pre``, ``h``, ``out``.
    """
    x = np.asarray(x, np.float64)
    if logits is None:
        logits = gate_logits(router_input(x, cfg)[0], w_gate, logit_bias)
    g = route(logits, cfg)
    rt = g["routing"]
    x_disp = dispatch(x, rt)
    h_pre, h, out = expert_ffn(x_disp, rt.offsets, w1, b1, w2, b2, cfg.act)
    y = combine(out, rt, g["weights"], x.shape[1])
    g.update(x_disp=x_disp, h_pre=h_pre, h=h, out=out, y=y)
    return g


def dense_mixture(cfg: LayerConfig, x, w_gate, w1, b1, w2, b2, logit_bias=None):
    """Capacity-free dense form: every expert runs on every token and the
    outputs are mixed by the top-k weights (zero off the top-k)
    ([DeepSeek-MoE traps] ch.1 ``moe_forward``; [deepspeed.moe overview]
    §6.5 compare MoE against a dense computation).  Equals ``forward`` when
    ``drop_tokens`` is false."""
    x = np.asarray(x, np.float64)
    lg = gate_logits(router_input(x, cfg)[0], w_gate, logit_bias)
    p = softmax(lg / cfg.gate_temperature)
    idx = select_experts(lg, cfg)
    w = gate_weights(p, idx)
    S, E = lg.shape
    mix = np.zeros((S, E), np.float64)
    np.put_along_axis(mix, idx, w, axis=1)
    y = np.zeros_like(x)
    for e in range(E):
        he = activation(x @ np.asarray(w1[e], np.float64).T + np.asarray(b1[e], np.float64), cfg.act)
        ye = he @ np.asarray(w2[e], np.float64).T + np.asarray(b2[e], np.float64)
        y += mix[:, e:e + 1] * ye
    return y


def residual_mlp(x, rw1, rb1, rw2, rb2, act: str) -> np.ndarray:
    """PR-MoE's fixed MLP on every token ([deepspeed.moe overview] §2.3 and
    §3.3: ``use_residual=True`` combines a fixed MLP with the dynamic
    experts): act(x rw1^T + rb1) rw2^T + rb2, the shape of one expert."""
    x = np.asarray(x, np.float64)
    h = activation(x @ np.asarray(rw1, np.float64).T + np.asarray(rb1, np.float64), act)
    return h @ np.asarray(rw2, np.float64).T + np.asarray(rb2, np.float64)


def residual_coef(x, coef_w, coef_b) -> np.ndarray:
    """Per-token mixing weights of the two branches (reading R8, second
    form): c[s] = softmax over 2 of (x_s W_c^T + b_c); W_c [2,d], b_c [2]."""
    z = np.asarray(x, np.float64) @ np.asarray(coef_w, np.float64).T + np.asarray(coef_b, np.float64)
    z = z - z.max(axis=1, keepdims=True)
    ez = np.exp(z)
    return ez / ez.sum(axis=1, keepdims=True)


def forward_residual(cfg: LayerConfig, x, w_gate, w1, b1, w2, b2, rw1, rb1, rw2, rb2,
                     logit_bias=None, logits: Optional[np.ndarray] = None,
                     coef_w=None, coef_b=None) -> dict:
    """The PR-MoE layer.  The page names the residual connection but gives no
    mixing formula; reading R8: the connection is a sum,
    y = MoE(x) + MLP(x), or, when the mixing weights W_c [2,d], b_c [2] are
    given, y = c0 MoE(x) + c1 MLP(x) with c = residual_coef(x, W_c, b_c).
    Returns ``forward``'s dict with ``y`` replaced and ``y_moe`` /
    ``residual`` (and ``coef``) added."""
    g = forward(cfg, x, w_gate, w1, b1, w2, b2, logit_bias=logit_bias, logits=logits)
    r = residual_mlp(x, rw1, rb1, rw2, rb2, cfg.act)
    g["y_moe"] = g["y"]
    g["residual"] = r
    if coef_w is None:
        g["y"] = g["y_moe"] + r
    else:
        c = residual_coef(x, coef_w, coef_b)
        g["coef"] = c
        g["y"] = c[:, 0:1] * g["y_moe"] + c[:, 1:2] * r
    return g


# ---------------------------------------------------------------------------
# backward
# ---------------------------------------------------------------------------
def backward(cfg: LayerConfig, fwd: dict, x, w_gate, w1, w2, dy) -> dict:
    """Gradients of L = <dY, y> + aux_loss_weight * l_aux.

    Routing (top-k indices, slots, drops, first-choice counts) is a constant
    of the backward pass ([DeepSeek-MoE traps] §3.1 ``TopKRouter``: the
    gradient is scattered only to the selected logits); an expert with no
    kept row gets dW = db = 0 written out ([DeepSeek-MoE traps] §2.1/§2.3).

    Chain, in order:
      dw[s,j]  = <dY_s, out[row(s,j)]>            (kept choices only)
      dO[row]  = w[s,j] * dY_s
      dW2_e    = sum_rows dO^T h,  db2_e = sum_rows dO
      dh_pre   = (dO W2_e) * act'(h_pre)
      dW1_e    = sum_rows dh_pre^T x_disp,  db1_e = sum_rows dh_pre
      dx_disp  = dh_pre W1_e
      dp       = d(weights)/dp applied to dw  (+ aux term E*first_e/S^2)
      dlogits  = p * (dp - <dp, p>)
      dW_g     = dlogits^T x,  dX = sum_j dx_disp[row(s,j)] + dlogits W_g
    """
    x = np.asarray(x, np.float64)
    dy = np.asarray(dy, np.float64)
    w_gate = np.asarray(w_gate, np.float64)
    rt: Routing = fwd["routing"]
    S, k = rt.idx.shape
    E, f, d = w1.shape
    w = fwd["weights"]
    p = fwd["probs"]
    out = fwd["out"]
    h = fwd["h"]
    h_pre = fwd["h_pre"]
    x_disp = fwd["x_disp"]
    R = rt.num_rows

    dw = np.zeros((S, k), np.float64)
    d_out = np.zeros((R, d), np.float64)
    for s in range(S):
        for j in range(k):
            r = rt.row_of(s, j)
            if r >= 0:
                dw[s, j] = float(dy[s] @ out[r])
                d_out[r] = w[s, j] * dy[s]

    dw1 = np.zeros((E, f, d), np.float64)
    db1 = np.zeros((E, f), np.float64)
    dw2 = np.zeros((E, d, f), np.float64)
    db2 = np.zeros((E, d), np.float64)
    dx_disp = np.zeros((R, d), np.float64)
    for e in range(E):
        a, b = int(rt.offsets[e]), int(rt.offsets[e + 1])
        if a == b:
            continue
        dO = d_out[a:b]
        dw2[e] = dO.T @ h[a:b]
        db2[e] = dO.sum(axis=0)
        dh_pre = (dO @ np.asarray(w2[e], np.float64)) * activation_grad(h_pre[a:b], cfg.act)
        dw1[e] = dh_pre.T @ x_disp[a:b]
        db1[e] = dh_pre.sum(axis=0)
        dx_disp[a:b] = dh_pre @ np.asarray(w1[e], np.float64)

    # weights -> probabilities (reading R2), then the aux-loss term (R5)
    dp = np.zeros((S, E), np.float64)
    rows = np.arange(S)
    if k == 1:
        dp[rows, rt.idx[:, 0]] += dw[:, 0]
    else:
        p1 = p[rows, rt.idx[:, 0]]
        p2 = p[rows, rt.idx[:, 1]]
        P2 = (p1 + p2) ** 2
        dp[rows, rt.idx[:, 0]] += p2 * (dw[:, 0] - dw[:, 1]) / P2
        dp[rows, rt.idx[:, 1]] += p1 * (dw[:, 1] - dw[:, 0]) / P2
    if cfg.aux_loss_weight != 0.0:
        if cfg.aux_loss_type == "std":
            # d std(u) / d p[s,e] = (u_e - mean u) / (E * std u) * 1/S
            u = p.mean(axis=0)
            sd = np.sqrt(np.mean((u - u.mean()) ** 2))
            if sd > 0.0:
                dp += cfg.aux_loss_weight * ((u - u.mean()) / (E * S * sd))[None, :]
        else:
            first = np.bincount(rt.idx[:, 0], minlength=E).astype(np.float64)
            dp += cfg.aux_loss_weight * E * first[None, :] / float(S * S)

    # p = softmax(logits / T): the logits' gradient carries the 1/T
    dlogits = p * (dp - np.sum(dp * p, axis=1, keepdims=True)) / cfg.gate_temperature
    # the router saw x~ = x * f under jitter (R12)
    xr, jf = router_input(x, cfg)
    dw_gate = dlogits.T @ xr
    dx = dlogits @ w_gate
    if jf is not None:
        dx = dx * jf.astype(np.float64)
    for s in range(S):
        for j in range(k):
            r = rt.row_of(s, j)
            if r >= 0:
                dx[s] += dx_disp[r]
    return {"dx": dx, "dw1": dw1, "db1": db1, "dw2": dw2, "db2": db2,
            "dw_gate": dw_gate, "dlogits": dlogits, "dw": dw, "d_out": d_out,
            "dx_disp": dx_disp}


def loss(cfg: LayerConfig, x, w_gate, w1, b1, w2, b2, dy, logit_bias=None,
         routing_from: Optional[dict] = None) -> float:
    """Scalar L = <dY, y> + aux_loss_weight * l_aux, used by finite-difference
    checks.  ``routing_from`` freezes routing (indices, slots, first-choice
    counts) to that of a previous forward, so that a perturbation cannot move
    a token between experts."""
    x = np.asarray(x, np.float64)
    lg = gate_logits(router_input(x, cfg)[0], w_gate, logit_bias)
    p = softmax(lg / cfg.gate_temperature)
    if routing_from is None:
        g = route(lg, cfg)
        rt, idx = g["routing"], g["routing"].idx
    else:
        rt = routing_from["routing"]
        idx = rt.idx
    w = gate_weights(p, idx)
    x_disp = dispatch(x, rt)
    _, _, out = expert_ffn(x_disp, rt.offsets, w1, b1, w2, b2, cfg.act)
    y = combine(out, rt, w, x.shape[1])
    val = float(np.sum(np.asarray(dy, np.float64) * y))
    if cfg.aux_loss_weight != 0.0:
        val += cfg.aux_loss_weight * aux_loss(p, idx, cfg.aux_loss_type)
    return val
