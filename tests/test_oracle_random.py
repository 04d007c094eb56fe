"""Pins of the oracle's in-layer randomness (gating variants R11-R14): the
Philox4x32-10 generator against its published known-answer vectors, the
uniform / Gumbel / jitter transforms against closed forms, distributions and
IEEE float32 arithmetic done by torch, the random-token-selection
permutation (a bijection, its queue order checked by a brute-force count),
the Gumbel-max choice against the softmax probabilities it must sample, and
the backward under jitter by central finite differences."""
import math

import numpy as np
import pytest
import torch
from scipy import stats
from scipy.special import softmax as scipy_softmax

from oracle import moe_oracle as O
from oracle import random_streams as RS


# --------------------------------------------------------------------------
# Philox4x32-10
# --------------------------------------------------------------------------
@pytest.mark.parametrize("ctr,key,want", [
    # known-answer vectors published with the Random123 reference
    # implementation of Salmon et al. (SC 2011)
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF, 0xFFFFFFFF),
     (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
])
def test_philox_known_answers(ctr, key, want):
    got = RS.philox4x32_10(*ctr, *key)
    assert tuple(int(v) for v in got) == want


def test_philox_vectorises_like_single_calls():
    rng = np.random.default_rng(1)
    c = rng.integers(0, 2 ** 32, size=(4, 50), dtype=np.uint64)
    out = RS.philox4x32_10(c[0], c[1], c[2], c[3], 0x1234, 0xABCD)
    for i in range(50):
        one = RS.philox4x32_10(int(c[0, i]), int(c[1, i]), int(c[2, i]), int(c[3, i]),
                               0x1234, 0xABCD)
        assert tuple(int(o[i]) for o in out) == tuple(int(v) for v in one)


# --------------------------------------------------------------------------
# streams and transforms
# --------------------------------------------------------------------------
def test_uniform_is_open_interval_and_float32_exact():
    u = RS.uniform_open(np.array([0, 511, 512, 0xFFFFFFFF], dtype=np.uint64))
    assert u[0] == 2.0 ** -24 and u[1] == 2.0 ** -24      # the 9 low bits are dropped
    assert u[2] == 3 * 2.0 ** -24
    assert u[3] == 1.0 - 2.0 ** -24
    w = np.random.default_rng(2).integers(0, 2 ** 32, 10000, dtype=np.uint64)
    uu = RS.uniform_open(w)
    assert np.all(uu.astype(np.float32).astype(np.float64) == uu)
    assert np.all((uu > 0) & (uu < 1))


def test_stream_layout_and_uniformity():
    S, E = 300, 10
    u = RS.stream_uniforms(S, E, RS.PURPOSE_GATE_NOISE, seed=(7 << 32) | 3, offset=(5 << 32) | 9)
    # element (s, e) is word e % 4 of the counter (s, 1 << 24 | e // 4, offset lo, offset hi)
    for s, e in [(0, 0), (1, 5), (299, 9), (17, 3), (42, 8)]:
        w = RS.philox4x32_10(s, (1 << 24) | (e // 4), 9, 5, 3, 7)[e % 4]
        assert u[s, e] == RS.uniform_open(w)
    assert stats.kstest(u.ravel(), "uniform").pvalue > 1e-4
    # a different purpose, offset or seed is a different stream
    other = [RS.stream_uniforms(S, E, RS.PURPOSE_JITTER, (7 << 32) | 3, (5 << 32) | 9),
             RS.stream_uniforms(S, E, RS.PURPOSE_GATE_NOISE, (7 << 32) | 3, (5 << 32) | 10),
             RS.stream_uniforms(S, E, RS.PURPOSE_GATE_NOISE, (7 << 32) | 4, (5 << 32) | 9)]
    for o in other:
        assert np.mean(o == u) < 0.01


def test_gumbel_closed_forms_and_moments():
    for x in (-1.5, 0.0, 0.7, 3.0):
        assert abs(RS.gumbel(np.exp(-np.exp(-x))) - x) < 1e-12
    _, g = RS.gate_noise(20000, 8, seed=11, offset=0)
    n = g.size
    assert abs(g.mean() - np.euler_gamma) < 6 * math.sqrt(math.pi ** 2 / 6 / n)
    assert abs(g.var() - math.pi ** 2 / 6) < 0.05
    assert stats.kstest(g.ravel(), "gumbel_r").pvalue > 1e-4


def test_jitter_factors_are_float32_arithmetic():
    eps = 0.01
    f = RS.jitter_factors(64, 40, eps, seed=5, offset=2)
    u = torch.from_numpy(RS.stream_uniforms(64, 40, RS.PURPOSE_JITTER, 5, 2)).float()
    ref = 1.0 + torch.tensor(eps, dtype=torch.float32) * (2.0 * u - 1.0)   # torch float32 ops
    assert f.dtype == np.float32 and np.array_equal(f, ref.numpy())
    assert np.all((f >= 1 - eps) & (f <= 1 + eps))
    assert abs(float(f.mean()) - 1.0) < 1e-3


def test_router_input_under_jitter():
    rng = np.random.default_rng(4)
    x = torch.randn(33, 24, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    xd = x.double().numpy()
    c = O.LayerConfig(33, 24, 8, 4, 2, 1.0, 1, True, "relu", noise_policy="jitter",
                      noise_seed=9, noise_offset=1)
    xr, f = O.router_input(xd, c)
    want = (x.float() * torch.from_numpy(f)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(xr, want)
    c.dtype = "f32"
    xr32, _ = O.router_input(xd, c)
    assert np.array_equal(xr32, (x.float() * torch.from_numpy(f)).double().numpy())
    c.noise_policy = "none"
    same, none = O.router_input(xd, c)
    assert none is None and np.array_equal(same, xd)
    del rng


# --------------------------------------------------------------------------
# the choice: Gumbel-max samples the softmax
# --------------------------------------------------------------------------
def test_rsample_choice_samples_the_softmax():
    """With the same logits row for every token, the top-1 of logits + g is a
    sample of softmax(logits): its frequencies match the probabilities."""
    S, E = 40000, 5
    row = np.array([1.0, 0.2, -0.5, 0.9, -2.0])
    c = O.LayerConfig(S, 8, 8, E, 1, 1.0, 1, False, "relu", noise_policy="rsample",
                      noise_seed=123, noise_offset=0)
    idx = O.select_experts(np.tile(row, (S, 1)), c)
    freq = np.bincount(idx[:, 0], minlength=E) / S
    p = scipy_softmax(row)
    assert np.all(np.abs(freq - p) < 6 * np.sqrt(p * (1 - p) / S))


def test_second_expert_sampling():
    """First choice: the noise-free arg-max, always.  Second: a sample of the
    softmax over the other experts."""
    S, E = 40000, 4
    row = np.array([0.3, 2.0, -0.4, 0.8])
    c = O.LayerConfig(S, 8, 8, E, 2, 1.0, 1, False, "relu", second_expert_sampling=True,
                      noise_seed=77, noise_offset=3)
    idx = O.select_experts(np.tile(row, (S, 1)), c)
    assert np.all(idx[:, 0] == 1)
    assert np.all(idx[:, 1] != 1)
    freq = np.bincount(idx[:, 1], minlength=E) / S
    rest = row.copy()
    rest[1] = -np.inf
    p = scipy_softmax(rest)
    assert np.all(np.abs(freq - p) < 6 * np.sqrt(p * (1 - p) / S) + 1e-12)


def test_rsample_keys_are_float32_sums():
    """The choice compares the float32 sums logit + g: two experts whose
    float64 sums differ but whose float32 sums tie go to the lower index."""
    c = O.LayerConfig(1, 8, 8, 2, 1, 1.0, 1, False, "relu", noise_policy="rsample")
    lg = np.array([[1.0, 1.0 + 2.0 ** -30]])
    g = np.zeros((1, 2))
    assert O.select_experts(lg, c, g)[0, 0] == 0          # ties in float32
    assert O.topk_experts(lg, 1)[0, 0] == 1               # not in float64


@pytest.mark.parametrize("opts", [dict(), dict(noise_policy="jitter"), dict(use_rts=True),
                                  dict(second_expert_sampling=True)])
def test_noise_leaves_the_choice_alone_unless_an_option_reads_it(opts):
    """Only rsample and second-expert sampling with k = 2 choose on Gumbel
    keys; jitter, random token selection and k = 1 choose on the logits
    whatever noise is passed."""
    k = 1 if opts.get("second_expert_sampling") else 2
    c = O.LayerConfig(64, 8, 8, 4, k, 1.0, 1, True, "relu", **opts)
    rng = np.random.default_rng(5)
    lg = rng.standard_normal((64, 4))
    g = 50.0 * rng.standard_normal((64, 4))               # would reorder almost every row
    assert np.array_equal(O.select_experts(lg, c, g), O.topk_experts(lg, k))
    assert np.array_equal(O.route(lg, c, noise=g)["routing"].idx, O.topk_experts(lg, k))


# --------------------------------------------------------------------------
# random token selection
# --------------------------------------------------------------------------
@pytest.mark.parametrize("S", [1, 2, 3, 5, 17, 100, 1000, 4097, 16384])
def test_rts_permutation_is_a_bijection(S):
    pi = RS.rts_position(S, seed=31, offset=7)
    assert sorted(pi.tolist()) == list(range(S))
    assert np.array_equal(pi, RS.rts_position(S, seed=31, offset=7))
    if S >= 100:
        assert not np.array_equal(pi, RS.rts_position(S, seed=32, offset=7))
        assert not np.array_equal(pi, RS.rts_position(S, seed=31, offset=8))
        assert np.mean(pi == np.arange(S)) < 0.05


def test_rts_position_of_a_token_is_uniform_over_seeds():
    S, n = 6, 6000
    first = np.array([RS.rts_position(S, seed=s, offset=0)[0] for s in range(n)])
    counts = np.bincount(first, minlength=S)
    assert stats.chisquare(counts).pvalue > 1e-4


def brute_force_rts_slots(idx, pos):
    """slot(s, j) = #{(s', j') with the same expert, (j', pi(s')) < (j, pi(s))}."""
    S, k = idx.shape
    slot = np.zeros((S, k), np.int64)
    for s in range(S):
        for j in range(k):
            slot[s, j] = sum(1 for s2 in range(S) for j2 in range(k)
                             if idx[s2, j2] == idx[s, j] and (j2, pos[s2]) < (j, pos[s]))
    return slot


@pytest.mark.parametrize("k", [1, 2])
def test_rts_slots_brute_force(k):
    rng = np.random.default_rng(60 + k)
    S, E = 40, 4
    lg = rng.standard_normal((S, E))
    c = O.LayerConfig(S, 8, 8, E, k, 0.5, 1, True, "relu", use_rts=True, noise_seed=5,
                      noise_offset=k)
    g = O.route(lg, c)
    rt = g["routing"]
    pos = RS.rts_position(S, 5, k)
    full = brute_force_rts_slots(rt.idx, pos)
    cap = rt.capacity
    assert np.array_equal(rt.slot, np.where(full < cap, full, -1))
    assert (rt.slot < 0).any()
    # the kept first choices of an expert are the ones earliest in the queue
    for e in range(E):
        toks = np.nonzero(rt.idx[:, 0] == e)[0]
        kept = set(toks[rt.slot[toks, 0] >= 0].tolist())
        want = set(sorted(toks.tolist(), key=lambda t: pos[t])[:min(cap, len(toks))])
        assert kept == want
    # without RTS the same logits give token-order slots
    c.use_rts = False
    plain = O.route(lg, c)["routing"]
    assert np.array_equal(plain.slot, np.where(brute_force_rts_slots(rt.idx, np.arange(S)) < cap,
                                               brute_force_rts_slots(rt.idx, np.arange(S)), -1))


# --------------------------------------------------------------------------
# backward under the noise options
# --------------------------------------------------------------------------
@pytest.mark.parametrize("policy,second,rts", [("jitter", False, False), ("rsample", False, True),
                                               ("none", True, True)])
def test_backward_finite_differences_with_noise(policy, second, rts):
    rng = np.random.default_rng(70)
    S, d, f, E, k = 7, 4, 5, 4, 2
    c = O.LayerConfig(S, d, f, E, k, 0.5, 1, True, O.ACT_GELU_TANH, aux_loss_weight=0.05,
                      noise_policy=policy, second_expert_sampling=second, use_rts=rts,
                      noise_seed=3, noise_offset=4, jitter_eps=0.2, dtype="f64")
    x = rng.standard_normal((S, d))
    wg = rng.standard_normal((E, d)) * 0.7
    w1, b1 = rng.standard_normal((E, f, d)) * 0.5, rng.standard_normal((E, f)) * 0.3
    w2, b2 = rng.standard_normal((E, d, f)) * 0.5, rng.standard_normal((E, d)) * 0.3
    dy = rng.standard_normal((S, d))
    fwd = O.forward(c, x, wg, w1, b1, w2, b2)
    g = O.backward(c, fwd, x, wg, w1, w2, dy)
    h = 1e-6

    def L(**over):
        a = dict(x=x, w_gate=wg, w1=w1, b1=b1, w2=w2, b2=b2)
        a.update(over)
        return O.loss(c, a["x"], a["w_gate"], a["w1"], a["b1"], a["w2"], a["b2"], dy,
                      routing_from=fwd)

    for name, arr, grad in [("x", x, g["dx"]), ("w_gate", wg, g["dw_gate"])]:
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            ap, am = arr.copy(), arr.copy()
            ap[i] += h
            am[i] -= h
            num[i] = (L(**{name: ap}) - L(**{name: am})) / (2 * h)
        assert np.allclose(grad, num, rtol=1e-6, atol=1e-7), name
