"""Pins of the float64 oracle to facts other than itself.

Each test checks the oracle against something written independently of it:
the pages' worked capacity arithmetic (tests/golden/capacity_pages.json),
hand-worked routing cases, brute-force enumeration under a different
formulation, library routines (scipy softmax, torch GELU/linear), closed-form
special cases, dense equivalence and central finite differences.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax as scipy_softmax

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def cfg(S, d, f, E, k, cf=1.0, min_cap=1, drop=True, act=O.ACT_GELU_TANH, aux=0.0):
    return O.LayerConfig(S, d, f, E, k, cf, min_cap, drop, act, aux)


# --------------------------------------------------------------------------
# capacity
# --------------------------------------------------------------------------
def test_capacity_pages_worked_arithmetic():
    data = json.load(open(os.path.join(GOLDEN, "capacity_pages.json")))
    for c in data["cases"]:
        got = O.capacity(c["S"], c["E"], c["k"], c["cf"], c["min_capacity"], True)
        assert got == c["expected"], c["cite"]


@pytest.mark.parametrize("S,E,k,cf,expected", [
    (256, 4, 1, 1.0, 64),        # tiny fp32 layer
    (4096, 8, 2, 1.0, 1024),     # 8 experts
    (16384, 64, 2, 1.25, 640),   # 64 experts: ceil(16384*2/64*1.25)
    (8192, 16, 2, 2.0, 2048),    # skewed, capped
    (8192, 32, 2, 1.25, 640),    # training layer
])
def test_capacity_of_the_layer_configs(S, E, k, cf, expected):
    assert O.capacity(S, E, k, cf, 4, True) == expected


def test_capacity_ceil_min_and_exact_decimal():
    # ceil, not floor: 10*1/4 = 2.5 -> 3 (the cf=1.25 formula is a ceiling)
    assert O.capacity(10, 4, 1, 1.0, 1, True) == 3
    # min_capacity binds: 8/4 = 2 < 4
    assert O.capacity(8, 4, 1, 1.0, 4, True) == 4
    # 100 * 1.1 is exactly 110; binary floating point gives 110.00000000000001
    assert O.capacity(100, 1, 1, 1.1, 1, True) == 110
    assert math.ceil(100 * 1.1) == 111
    assert O.capacity(100, 1, 1, 1.1, 1, False) is None


# --------------------------------------------------------------------------
# top-k
# --------------------------------------------------------------------------
def brute_force_topk(row, k):
    """Different formulation: the k-subset with the largest logit sum, the
    lexicographically smallest sorted index tuple among equal sums, ordered
    by logit descending then index ascending."""
    E = len(row)
    best = None
    for comb in itertools.combinations(range(E), k):
        key = (-sum(row[c] for c in comb), comb)
        if best is None or key < best:
            best = key
    chosen = sorted(best[1], key=lambda c: (-row[c], c))
    return chosen


def test_topk_brute_force_with_many_ties():
    rng = np.random.default_rng(0)
    for E in (1, 2, 3, 5, 8):
        for k in (1, 2):
            if k > E:
                continue
            lg = rng.integers(0, 3, size=(200, E)).astype(np.float64)
            idx = O.topk_experts(lg, k)
            for s in range(lg.shape[0]):
                assert list(idx[s]) == brute_force_topk(list(lg[s]), k)


def test_topk_continuous_matches_stable_argsort():
    rng = np.random.default_rng(1)
    lg = rng.standard_normal((500, 16))
    idx = O.topk_experts(lg, 2)
    ref = np.argsort(-lg, axis=1, kind="stable")[:, :2]
    assert np.array_equal(idx, ref)


def test_exact_tie_cases():
    assert O.topk_experts(np.array([[1.0, 1.0, 0.0]]), 2).tolist() == [[0, 1]]
    assert O.topk_experts(np.array([[0.0, 1.0, 1.0]]), 2).tolist() == [[1, 2]]
    assert O.topk_experts(np.array([[2.0, 2.0, 2.0, 2.0]]), 2).tolist() == [[0, 1]]
    p = O.softmax(np.array([[1.0, 1.0, 0.0]]))
    w = O.gate_weights(p, np.array([[0, 1]]))
    assert w.tolist() == [[0.5, 0.5]]


# --------------------------------------------------------------------------
# gate logits
# --------------------------------------------------------------------------
def test_gate_logits_against_torch_linear():
    """logits = x W_g^T + b is torch's Linear layer (the router of the MoE
    explainer §3.1 Step 1) in float64: without a bias, with one [E] bias
    shared by every token, and with a per-token [S,E] bias (caller-drawn
    gate noise) added row by row."""
    rng = np.random.default_rng(41)
    S, d, E = 37, 24, 5
    x = rng.standard_normal((S, d))
    w = rng.standard_normal((E, d))
    b = rng.standard_normal(E)
    B = rng.standard_normal((S, E))
    tx, tw = torch.from_numpy(x), torch.from_numpy(w)
    lin = torch.nn.functional.linear
    assert np.allclose(O.gate_logits(x, w), lin(tx, tw).numpy(), rtol=1e-13, atol=1e-13)
    assert np.allclose(O.gate_logits(x, w, b), lin(tx, tw, torch.from_numpy(b)).numpy(),
                       rtol=1e-13, atol=1e-13)
    per_tok = torch.stack([lin(tx[s], tw, torch.from_numpy(B[s])) for s in range(S)])
    assert np.allclose(O.gate_logits(x, w, B), per_tok.numpy(), rtol=1e-13, atol=1e-13)


def test_gate_logits_bias_forms_are_local():
    """A per-token bias moves only its own token's logit; an [E] bias moves
    that expert's logit of every token by the same amount; the operand is
    x W_g^T, not x W_g or W_g x (a transposed weight fails the shape or the
    single-entry check)."""
    rng = np.random.default_rng(42)
    S, d, E = 6, 4, 3
    x = rng.standard_normal((S, d))
    w = rng.standard_normal((E, d))
    base = O.gate_logits(x, w)
    B = np.zeros((S, E))
    B[4, 1] = 2.5
    diff = O.gate_logits(x, w, B) - base
    want = np.zeros((S, E))
    want[4, 1] = 2.5
    assert np.allclose(diff, want, rtol=0, atol=1e-14)
    b = np.array([0.0, -1.0, 0.5])
    assert np.allclose(O.gate_logits(x, w, b) - base, np.tile(b, (S, 1)), rtol=0, atol=1e-14)
    # one-hot token and one-hot weight row pick out a single weight entry
    xo = np.zeros((1, d))
    xo[0, 3] = 1.0
    assert np.allclose(O.gate_logits(xo, w)[0], w[:, 3], rtol=0, atol=0)


# --------------------------------------------------------------------------
# softmax / weights / l_aux
# --------------------------------------------------------------------------
def test_softmax_matches_scipy():
    rng = np.random.default_rng(2)
    lg = rng.standard_normal((64, 7)) * 5
    assert np.allclose(O.softmax(lg), scipy_softmax(lg, axis=1), rtol=0, atol=1e-15)


def test_weights_k2_is_softmax_over_selected_logits():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((300, 6))
    idx = O.topk_experts(lg, 2)
    w = O.gate_weights(O.softmax(lg), idx)
    sel = np.take_along_axis(lg, idx, axis=1)
    ref = np.exp(sel) / np.exp(sel).sum(axis=1, keepdims=True)
    assert np.allclose(w, ref, rtol=1e-14, atol=0)
    assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    assert np.all(w > 0) and np.all(w <= 1)
    assert np.all(w[:, 0] >= w[:, 1])


def test_weights_k1_is_raw_probability():
    lg = np.array([[0.0, math.log(3.0)]])
    w = O.gate_weights(O.softmax(lg), O.topk_experts(lg, 1))
    assert abs(w[0, 0] - 0.75) < 1e-15


def test_gate_temperature_softmax_and_routing():
    """p = softmax(logits / T) (scipy), the top-k choice is the T = 1 choice,
    and the k=2 weights are the selected probabilities renormalised."""
    rng = np.random.default_rng(31)
    lg = rng.standard_normal((40, 6)) * 2.0
    for T in (0.5, 2.0):
        c = cfg(40, 8, 8, 6, 2, cf=2.0)
        c.gate_temperature = T
        g = O.route(lg, c)
        assert np.allclose(g["probs"], scipy_softmax(lg / T, axis=1), rtol=1e-13, atol=1e-15)
        g1 = O.route(lg, cfg(40, 8, 8, 6, 2, cf=2.0))
        assert np.array_equal(g["routing"].idx, g1["routing"].idx)
        ps = np.take_along_axis(scipy_softmax(lg / T, axis=1), g["routing"].idx, axis=1)
        assert np.allclose(g["weights"], ps / ps.sum(axis=1, keepdims=True), rtol=1e-13)


def test_std_balance_loss_hand_worked():
    """usage u = mean_s p = (0.7, 0.3): population std 0.2, l_aux = 0.2 + 1e-6;
    uniform probabilities give std 0, l_aux = 1e-6."""
    p = np.array([[0.9, 0.1], [0.5, 0.5]])
    idx = np.array([[0], [0]])
    assert abs(O.aux_loss(p, idx, "std") - (0.2 + 1e-6)) < 1e-15
    u = np.full((5, 4), 0.25)
    assert O.aux_loss(u, np.zeros((5, 1), np.int64), "std") == 1e-6


def test_aux_loss_closed_forms():
    # uniform probabilities -> 1 whatever the first choices are
    assert abs(O.aux_loss(np.full((10, 4), 0.25), np.zeros((10, 1), np.int64)) - 1.0) < 1e-15
    # every token certain of expert 0 -> E
    lg = np.zeros((9, 5))
    lg[:, 0] = 1000.0
    p = O.softmax(lg)
    assert O.aux_loss(p, O.topk_experts(lg, 2)) == 5.0
    # hand-worked: p rows (1/4, 3/4), both first on expert 1 -> 2*(3/4*1) = 1.5
    lg = np.array([[0.0, math.log(3.0)]] * 2)
    p = O.softmax(lg)
    assert abs(O.aux_loss(p, O.topk_experts(lg, 2)) - 1.5) < 1e-15


# --------------------------------------------------------------------------
# slots and drops
# --------------------------------------------------------------------------
def brute_force_slots(idx, cap):
    """slot(s,j) = number of (s',j') on the same expert that come first in
    priority order (j' < j, or j' == j and s' < s); dropped if >= cap."""
    S, k = idx.shape
    slot = np.full((S, k), -1, np.int64)
    for s in range(S):
        for j in range(k):
            n = 0
            for s2 in range(S):
                for j2 in range(k):
                    if idx[s2, j2] == idx[s, j] and (j2 < j or (j2 == j and s2 < s)):
                        n += 1
            if cap is None or n < cap:
                slot[s, j] = n
    return slot


HAND_CASES = [
    # (i) 8 tokens all preferring expert 0, C = ceil(8*1*1/2) = 4
    dict(logits=[[1, 0]] * 8, k=1, cf=1.0, min_cap=1, cap=4,
         slot=[[0], [1], [2], [3], [-1], [-1], [-1], [-1]], routed=[8, 0], kept=[4, 0]),
    # (ii) same with min_capacity 6 -> C = 6
    dict(logits=[[1, 0]] * 8, k=1, cf=1.0, min_cap=6, cap=6,
         slot=[[0], [1], [2], [3], [4], [5], [-1], [-1]], routed=[8, 0], kept=[6, 0]),
    # (iii) first choices [0,0,1,0], C = 4: expert 0 gets s0,s1,s3 then s2's second;
    #       expert 1 gets s2 first then the seconds of s0,s1,s3
    dict(logits=[[1, 0], [1, 0], [0, 1], [1, 0]], k=2, cf=1.0, min_cap=1, cap=4,
         slot=[[0, 1], [1, 2], [0, 3], [2, 3]], routed=[4, 4], kept=[4, 4]),
    # (iv) same with cf = 0.5 -> C = 2: s3 loses both choices
    dict(logits=[[1, 0], [1, 0], [0, 1], [1, 0]], k=2, cf=0.5, min_cap=1, cap=2,
         slot=[[0, 1], [1, -1], [0, -1], [-1, -1]], routed=[4, 4], kept=[2, 2]),
]


@pytest.mark.parametrize("case", HAND_CASES)
def test_hand_worked_routing(case):
    lg = np.array(case["logits"], np.float64)
    S, E = lg.shape
    c = cfg(S, 4, 4, E, case["k"], cf=case["cf"], min_cap=case["min_cap"])
    g = O.route(lg, c)
    rt = g["routing"]
    assert rt.capacity == case["cap"]
    assert rt.slot.tolist() == case["slot"]
    assert rt.routed.tolist() == case["routed"]
    assert rt.kept.tolist() == case["kept"]


def test_fully_dropped_token_outputs_zero():
    case = HAND_CASES[3]
    lg = np.array(case["logits"], np.float64)
    c = cfg(4, 3, 5, 2, 2, cf=0.5)
    rng = np.random.default_rng(4)
    x = rng.standard_normal((4, 3))
    w1, w2 = rng.standard_normal((2, 5, 3)), rng.standard_normal((2, 3, 5))
    b1, b2 = rng.standard_normal((2, 5)), rng.standard_normal((2, 3))
    out = O.forward(c, x, None, w1, b1, w2, b2, logits=lg)
    assert np.all(out["y"][3] == 0.0)
    assert np.any(out["y"][0] != 0.0)


@pytest.mark.parametrize("k", [1, 2])
def test_slots_brute_force_and_invariants(k):
    rng = np.random.default_rng(5 + k)
    for trial in range(30):
        S, E = int(rng.integers(1, 40)), int(rng.integers(max(k, 1), 6))
        lg = rng.integers(0, 4, size=(S, E)).astype(np.float64)
        cf = float(rng.choice([0.25, 0.5, 1.0, 2.0]))
        drop = bool(rng.integers(0, 2))
        c = cfg(S, 4, 4, E, k, cf=cf, min_cap=int(rng.integers(1, 4)), drop=drop)
        rt = O.route(lg, c)["routing"]
        assert np.array_equal(rt.slot, brute_force_slots(rt.idx, rt.capacity))
        # at most k kept per token; kept <= C; slots per expert are 0..routed-1
        assert np.all((rt.slot >= 0).sum(axis=1) <= k)
        if rt.capacity is not None:
            assert np.all(rt.kept <= rt.capacity)
        for e in range(E):
            mine = []
            for s in range(S):
                for j in range(k):
                    if rt.idx[s, j] == e:
                        mine.append((j, s))
            assert len(mine) == rt.routed[e]
            # priority order: every first choice's slot below every second's
            firsts = [s for (j, s) in mine if j == 0]
            seconds = [s for (j, s) in mine if j == 1]
            if firsts and seconds:
                f_slots = [rt.slot[s, 0] for s in firsts if rt.slot[s, 0] >= 0]
                s_slots = [rt.slot[s, 1] for s in seconds if rt.slot[s, 1] >= 0]
                if f_slots and s_slots:
                    assert max(f_slots) < min(s_slots)
        assert rt.num_rows == int(rt.kept.sum())
        # row_src is a bijection onto the kept (s, j) pairs
        pairs = sorted(int(v) for v in rt.row_src)
        kept_pairs = sorted(s * k + j for s in range(S) for j in range(k) if rt.slot[s, j] >= 0)
        assert pairs == kept_pairs


# --------------------------------------------------------------------------
# FFN, layer identities
# --------------------------------------------------------------------------
@pytest.mark.parametrize("act,tact", [(O.ACT_RELU, "relu"), (O.ACT_GELU_TANH, "tanh"),
                                      (O.ACT_GELU_ERF, "none")])
def test_expert_ffn_against_torch(act, tact):
    rng = np.random.default_rng(8)
    E, d, f = 3, 6, 10
    offsets = np.array([0, 4, 4, 9])
    xd = rng.standard_normal((9, d))
    w1, b1 = rng.standard_normal((E, f, d)), rng.standard_normal((E, f))
    w2, b2 = rng.standard_normal((E, d, f)), rng.standard_normal((E, d))
    h_pre, h, out = O.expert_ffn(xd, offsets, w1, b1, w2, b2, act)
    F = torch.nn.functional
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        xt = torch.from_numpy(xd[a:b])
        z = F.linear(xt, torch.from_numpy(w1[e]), torch.from_numpy(b1[e]))
        hz = F.relu(z) if tact == "relu" else F.gelu(z, approximate=tact)
        o = F.linear(hz, torch.from_numpy(w2[e]), torch.from_numpy(b2[e]))
        assert np.allclose(out[a:b], o.numpy(), rtol=1e-12, atol=1e-12)


def test_activation_grad_matches_torch_autograd():
    z = torch.linspace(-6, 6, 241, dtype=torch.float64, requires_grad=True)
    for act, tact in [(O.ACT_GELU_TANH, "tanh"), (O.ACT_GELU_ERF, "none")]:
        (g,) = torch.autograd.grad(torch.nn.functional.gelu(z, approximate=tact).sum(), z)
        assert np.allclose(O.activation_grad(z.detach().numpy(), act), g.numpy(),
                           rtol=1e-12, atol=1e-13)


def test_single_expert_is_plain_ffn():
    rng = np.random.default_rng(9)
    S, d, f = 12, 5, 7
    c = cfg(S, d, f, 1, 1, cf=1.0, min_cap=1)
    x = rng.standard_normal((S, d))
    wg = rng.standard_normal((1, d))
    w1, b1 = rng.standard_normal((1, f, d)), rng.standard_normal((1, f))
    w2, b2 = rng.standard_normal((1, d, f)), rng.standard_normal((1, d))
    y = O.forward(c, x, wg, w1, b1, w2, b2)["y"]
    ref = O.activation(x @ w1[0].T + b1[0], c.act) @ w2[0].T + b2[0]
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("act,tact", [(O.ACT_RELU, "relu"), (O.ACT_GELU_TANH, "tanh")])
def test_residual_layer_adds_a_dense_mlp(act, tact):
    """PR-MoE (reading R8): y_res - y_moe is torch's Linear -> act -> Linear
    on every token; zero residual weights give the plain layer exactly; with
    one expert, k=1 and the expert's weights as the residual's, y = 2 FFN(x)."""
    rng = np.random.default_rng(21)
    S, d, f, E = 30, 6, 9, 4
    c = cfg(S, d, f, E, 2, cf=0.75, min_cap=1, act=act)
    x = rng.standard_normal((S, d))
    wg = rng.standard_normal((E, d))
    w1, b1 = rng.standard_normal((E, f, d)), rng.standard_normal((E, f))
    w2, b2 = rng.standard_normal((E, d, f)), rng.standard_normal((E, d))
    rw1, rb1 = rng.standard_normal((f, d)), rng.standard_normal(f)
    rw2, rb2 = rng.standard_normal((d, f)), rng.standard_normal(d)
    g = O.forward_residual(c, x, wg, w1, b1, w2, b2, rw1, rb1, rw2, rb2)
    F = torch.nn.functional
    z = F.linear(torch.from_numpy(x), torch.from_numpy(rw1), torch.from_numpy(rb1))
    hz = F.relu(z) if tact == "relu" else F.gelu(z, approximate=tact)
    mlp = F.linear(hz, torch.from_numpy(rw2), torch.from_numpy(rb2)).numpy()
    assert np.allclose(g["y"] - g["y_moe"], mlp, rtol=1e-12, atol=1e-12)
    assert np.array_equal(g["y_moe"], O.forward(c, x, wg, w1, b1, w2, b2)["y"])
    zero = O.forward_residual(c, x, wg, w1, b1, w2, b2, rw1, rb1, np.zeros((d, f)), np.zeros(d))
    assert np.array_equal(zero["y"], zero["y_moe"])
    c1 = cfg(S, d, f, 1, 1, cf=1.0, min_cap=1, act=act)
    one = O.forward_residual(c1, x, wg[:1], w1[:1], b1[:1], w2[:1], b2[:1],
                             w1[0], b1[0], w2[0], b2[0])
    ffn = F.linear(F.relu(F.linear(torch.from_numpy(x), torch.from_numpy(w1[0]),
                                   torch.from_numpy(b1[0]))) if tact == "relu" else
                   F.gelu(F.linear(torch.from_numpy(x), torch.from_numpy(w1[0]),
                                   torch.from_numpy(b1[0])), approximate=tact),
                   torch.from_numpy(w2[0]), torch.from_numpy(b2[0])).numpy()
    assert np.allclose(one["y"], 2.0 * ffn, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("k", [1, 2])
def test_no_drop_equals_dense_mixture(k):
    rng = np.random.default_rng(10 + k)
    S, d, f, E = 40, 6, 9, 5
    c = cfg(S, d, f, E, k, cf=0.25, min_cap=1, drop=False)
    x = rng.standard_normal((S, d))
    wg = rng.standard_normal((E, d))
    w1, b1 = rng.standard_normal((E, f, d)), rng.standard_normal((E, f))
    w2, b2 = rng.standard_normal((E, d, f)), rng.standard_normal((E, d))
    bias = np.array([1.5, 0.0, -0.5, -2.0, 0.3])
    y = O.forward(c, x, wg, w1, b1, w2, b2, logit_bias=bias)["y"]
    ref = O.dense_mixture(c, x, wg, w1, b1, w2, b2, logit_bias=bias)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    # and with a tight capacity the two differ (tokens are dropped)
    c2 = cfg(S, d, f, E, k, cf=0.25, min_cap=1, drop=True)
    y2 = O.forward(c2, x, wg, w1, b1, w2, b2, logit_bias=bias)["y"]
    assert not np.allclose(y2, ref)


# --------------------------------------------------------------------------
# backward: central finite differences with routing held fixed
# --------------------------------------------------------------------------
def _fd_case(k, aux, drop, temp=1.0, aux_type="load", per_token=False):
    rng = np.random.default_rng(20 + 2 * k + int(drop))
    S, d, f, E = 7, 4, 5, 4
    c = cfg(S, d, f, E, k, cf=0.5 if drop else 1.0, min_cap=1, drop=drop, aux=aux)
    c.gate_temperature, c.aux_loss_type = temp, aux_type
    x = rng.standard_normal((S, d))
    wg = rng.standard_normal((E, d)) * 0.7
    w1, b1 = rng.standard_normal((E, f, d)) * 0.5, rng.standard_normal((E, f)) * 0.3
    w2, b2 = rng.standard_normal((E, d, f)) * 0.5, rng.standard_normal((E, d)) * 0.3
    bias = np.array([0.0, 0.4, 0.2, -30.0])     # expert 3 is never chosen
    dy = rng.standard_normal((S, d))
    if per_token:                                # noisy gating: per-token logit noise
        bias = bias[None, :] + 0.3 * rng.standard_normal((S, E))
    return c, x, wg, w1, b1, w2, b2, bias, dy


@pytest.mark.parametrize("k,aux,drop,temp,aux_type,per_token", [
    (1, 0.0, True, 1.0, "load", False), (2, 0.0, True, 1.0, "load", False),
    (2, 0.01, True, 1.0, "load", False), (2, 0.3, False, 1.0, "load", False),
    (1, 0.3, False, 1.0, "load", False),
    # gating variants: temperature, the std balance loss, per-token noise
    (2, 0.3, True, 0.5, "std", True), (1, 0.3, False, 2.0, "std", False),
    (2, 0.05, True, 0.5, "load", True)])
def test_backward_finite_differences(k, aux, drop, temp, aux_type, per_token):
    c, x, wg, w1, b1, w2, b2, bias, dy = _fd_case(k, aux, drop, temp, aux_type, per_token)
    fwd = O.forward(c, x, wg, w1, b1, w2, b2, logit_bias=bias)
    rt = fwd["routing"]
    if drop:
        assert (rt.slot < 0).any(), "case must drop something"
    # routing margins are far from ties so a 1e-6 step cannot flip them
    srt = np.sort(fwd["logits"], axis=1)[:, ::-1]
    assert np.min(srt[:, k - 1] - srt[:, k]) > 1e-3
    g = O.backward(c, fwd, x, wg, w1, w2, dy)
    h = 1e-6

    def L(**over):
        args = dict(x=x, w_gate=wg, w1=w1, b1=b1, w2=w2, b2=b2)
        args.update(over)
        return O.loss(c, args["x"], args["w_gate"], args["w1"], args["b1"], args["w2"],
                      args["b2"], dy, logit_bias=bias, routing_from=fwd)

    for name, arr, grad in [("x", x, g["dx"]), ("w_gate", wg, g["dw_gate"]),
                            ("w1", w1, g["dw1"]), ("b1", b1, g["db1"]),
                            ("w2", w2, g["dw2"]), ("b2", b2, g["db2"])]:
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            ap, am = arr.copy(), arr.copy()
            ap[i] += h
            am[i] -= h
            num[i] = (L(**{name: ap}) - L(**{name: am})) / (2 * h)
        assert np.allclose(grad, num, rtol=1e-6, atol=1e-7), name
    # the never-chosen expert gets exactly zero weight gradients
    assert rt.kept[3] == 0
    for key in ("dw1", "db1", "dw2", "db2"):
        assert np.all(g[key][3] == 0.0)


def test_residual_learned_mix_coefficient():
    """PR-MoE with learned per-token mixing (reading R8, second form): the two
    weights are a logistic sigmoid of the difference of two torch Linear
    outputs; zero mixing weights halve the sum form; a saturated bias gives
    the plain layer or the MLP alone."""
    from scipy.special import expit
    rng = np.random.default_rng(23)
    S, d, f, E = 25, 6, 8, 4
    c = cfg(S, d, f, E, 2, cf=1.0, min_cap=1)
    x = rng.standard_normal((S, d))
    wg = rng.standard_normal((E, d))
    w1, b1 = rng.standard_normal((E, f, d)), rng.standard_normal((E, f))
    w2, b2 = rng.standard_normal((E, d, f)), rng.standard_normal((E, d))
    rw1, rb1 = rng.standard_normal((f, d)), rng.standard_normal(f)
    rw2, rb2 = rng.standard_normal((d, f)), rng.standard_normal(d)
    cw, cb = rng.standard_normal((2, d)), rng.standard_normal(2)
    g = O.forward_residual(c, x, wg, w1, b1, w2, b2, rw1, rb1, rw2, rb2, coef_w=cw, coef_b=cb)
    z = torch.nn.functional.linear(torch.from_numpy(x), torch.from_numpy(cw),
                                   torch.from_numpy(cb)).numpy()
    c0 = expit(z[:, 0] - z[:, 1])
    assert np.allclose(g["coef"][:, 0], c0, rtol=1e-13, atol=1e-15)
    assert np.allclose(g["coef"][:, 1], 1.0 - c0, rtol=1e-12, atol=1e-15)
    plain = O.forward_residual(c, x, wg, w1, b1, w2, b2, rw1, rb1, rw2, rb2)
    assert np.allclose(g["y"], c0[:, None] * plain["y_moe"] + (1.0 - c0)[:, None] * plain["residual"],
                       rtol=1e-12, atol=1e-12)
    half = O.forward_residual(c, x, wg, w1, b1, w2, b2, rw1, rb1, rw2, rb2,
                              coef_w=np.zeros((2, d)), coef_b=np.zeros(2))
    assert np.allclose(half["y"], 0.5 * plain["y"], rtol=1e-14, atol=1e-14)
    for bias, want in (([40.0, -40.0], plain["y_moe"]), ([-40.0, 40.0], plain["residual"])):
        sat = O.forward_residual(c, x, wg, w1, b1, w2, b2, rw1, rb1, rw2, rb2,
                                 coef_w=np.zeros((2, d)), coef_b=np.array(bias))
        assert np.allclose(sat["y"], want, rtol=1e-12, atol=1e-12)
