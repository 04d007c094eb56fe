"""GPU routing parity: top-k, slots, drops, counts, offsets and row map are
bit-exact against the oracle fed the GPU's own fp32 logits; weights, probs,
logits and l_aux are within tolerance; disagreements of the oracle's own
float64 routing are only where the top-k margin is below 1e-4."""
import numpy as np
import pytest
import torch

from _harness import (DEV, GpuRun, WORKLOADS, check_routing_equal, f64, i64, oracle_cfg,
                      topk_margin)
from mixture_experts_layer_86_b300 import _native as N
from mixture_experts_layer_86_b300 import layer as L
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

FULL = ["tiny_fp32", "e8_bf16", "e64_bf16", "skew_e16_drop", "skew_e16_nodrop", "train_e32",
        "decode_e64"]


@pytest.mark.parametrize("name", FULL)
def test_routing_bit_exact_full_size(name):
    wl = WORKLOADS[name]
    run = GpuRun(wl, training=True)
    g = run.oracle_route()
    check_routing_equal(run, g)
    b = run.bufs
    assert np.allclose(f64(b["topk_w"]), g["weights"], rtol=2e-6, atol=1e-7)
    assert np.allclose(f64(b["probs"]), g["probs"], rtol=2e-6, atol=1e-8)
    assert abs(float(b["l_aux"].item()) - g["l_aux"]) <= 1e-5 * abs(g["l_aux"])
    if wl.k == 2:
        w = f64(b["topk_w"])
        assert np.allclose(w.sum(axis=1), 1.0, atol=1e-6)


@pytest.mark.parametrize("name", FULL)
def test_gate_logits_and_flip_audit(name):
    wl = WORKLOADS[name]
    run = GpuRun(wl)
    x = f64(run.inp.x)
    ref = O.gate_logits(x, f64(run.inp.w_gate),
                        None if run.inp.logit_bias is None else f64(run.inp.logit_bias))
    got = f64(run.bufs["logits"])
    err = np.abs(got - ref).max() / np.abs(ref).max()
    assert err <= 1e-5, err
    # the oracle's own routing vs the GPU's: flips only inside the 1e-4 margin
    own = O.topk_experts(ref, wl.k)
    gpu_idx = i64(run.bufs["topk_idx"])
    flips = np.nonzero(np.any(own != gpu_idx, axis=1))[0]
    margin = topk_margin(got, wl.k)
    assert np.all(margin[flips] < 1e-4), (len(flips), margin[flips].max() if len(flips) else 0)
    print(f"{name}: {len(flips)} routing flips, all with margin < 1e-4")


def _route_only(S, E, k, cf, min_cap, drop, logits):
    cfg = N.make_config(S, 8, 8, E, k, cf, min_cap, drop, "relu", "f32")
    R = max(N.moe_max_rows(cfg), 1)
    i32 = dict(dtype=torch.int32, device=DEV)
    out = {"probs": torch.empty((S, E), dtype=torch.float32, device=DEV),
           "topk_idx": torch.empty((S, k), **i32), "topk_w": torch.empty((S, k), dtype=torch.float32, device=DEV),
           "slot": torch.empty((S, k), **i32), "routed_cnt": torch.empty(E, **i32),
           "kept_cnt": torch.empty(E, **i32), "expert_offsets": torch.empty(E + 1, **i32),
           "row_src": torch.empty(R, **i32), "l_aux": torch.empty(1, dtype=torch.float32, device=DEV)}
    ws = L.alloc_workspace(cfg, DEV)
    lg = logits.to(DEV)
    N.moe_route_from_logits(cfg, lg, out["probs"], out["topk_idx"], out["topk_w"], out["slot"],
                            out["routed_cnt"], out["kept_cnt"], out["expert_offsets"],
                            out["row_src"], out["l_aux"], ws)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("S,E,k,cf,min_cap,drop", [
    (1, 2, 1, 1.0, 1, True), (129, 3, 2, 0.5, 1, True), (300, 5, 2, 1.0, 2, True),
    (1000, 8, 1, 0.75, 4, True), (4097, 16, 2, 1.25, 4, True), (513, 256, 2, 1.0, 1, True),
    (700, 64, 2, 2.0, 4, False), (256, 2, 2, 1.0, 4, True),
])
def test_route_with_exact_ties(S, E, k, cf, min_cap, drop):
    """Integer-valued logits: many exact ties, which must go to the lower
    index exactly as the oracle breaks them."""
    gen = torch.Generator().manual_seed(S * 31 + E)
    logits = torch.randint(0, 3, (S, E), generator=gen).float()
    out = _route_only(S, E, k, cf, min_cap, drop, logits)
    g = O.route(logits.double().numpy(), O.LayerConfig(S, 8, 8, E, k, cf, min_cap, drop, "relu"))
    rt = g["routing"]
    assert np.array_equal(i64(out["topk_idx"]), rt.idx)
    assert np.array_equal(i64(out["slot"]), rt.slot)
    assert np.array_equal(i64(out["routed_cnt"]), rt.routed)
    assert np.array_equal(i64(out["kept_cnt"]), rt.kept)
    assert np.array_equal(i64(out["expert_offsets"]), rt.offsets)
    assert np.array_equal(i64(out["row_src"])[:rt.num_rows], rt.row_src)
    assert np.allclose(f64(out["topk_w"]), g["weights"], rtol=2e-6)
    assert abs(float(out["l_aux"].item()) - g["l_aux"]) <= 1e-5 * max(abs(g["l_aux"]), 1e-12)


def test_route_hand_worked_case():
    """S=4, E=2, k=2, C=2: s3 loses both choices (worked by hand)."""
    logits = torch.tensor([[1.0, 0.0], [1.0, 0.0], [0.0, 1.0], [1.0, 0.0]])
    out = _route_only(4, 2, 2, 0.5, 1, True, logits)
    assert i64(out["slot"]).tolist() == [[0, 1], [1, -1], [0, -1], [-1, -1]]
    assert i64(out["kept_cnt"]).tolist() == [2, 2]
    assert i64(out["routed_cnt"]).tolist() == [4, 4]
    assert i64(out["expert_offsets"]).tolist() == [0, 2, 4]


@pytest.mark.parametrize("S", [18000, 20000])
def test_gate_routing_beyond_one_wave(S):
    """The single-launch bf16 gate takes one tile of at most 128 tokens per
    SM: 18000 tokens are 141 tiles of 128 (ragged last tile) on a 148-SM
    B300; 20000 tokens need more than one tile per SM, so the gate runs as
    three launches (fused gate kernel, slot scan, slot assignment).  Routing
    must match the oracle on the GPU's own logits either way."""
    wl = WORKLOADS["e8_bf16"].scaled(S)
    wl = type(wl)(**{**wl.__dict__, "hidden_size": 2048, "ffn_size": 64, "name": f"gate_S{S}"})
    run = GpuRun(wl, training=True)
    g = run.oracle_route()
    check_routing_equal(run, g)
    b = run.bufs
    assert np.allclose(f64(b["topk_w"]), g["weights"], rtol=2e-6, atol=1e-7)
    assert np.allclose(f64(b["probs"]), g["probs"], rtol=2e-6, atol=1e-8)
    assert abs(float(b["l_aux"].item()) - g["l_aux"]) <= 1e-5 * abs(g["l_aux"])
    assert N.moe_get_device_error() == 0


@pytest.mark.parametrize("S", [8192, 8449, 12000])
@pytest.mark.parametrize("base", ["e8_bf16", "tiny_fp32"])
def test_routing_scan_256_experts(base, S):
    """The routing scan at the widest expert count: with E = 256, k = 2 the
    512 count columns and 256 probability columns leave only 2 and 4 thread
    groups per column, each summing a run of 128-token CTAs.  8192 tokens
    (64 CTAs), 8449 (67, one token in the last CTA) and 12000 (94, ragged);
    routing must match the oracle on the GPU's own logits."""
    wl = WORKLOADS[base].scaled(S, bias_std=0.05)
    wl = type(wl)(**{**wl.__dict__, "num_experts": 256, "k": 2, "hidden_size": 256,
                     "ffn_size": 64, "name": f"scan256_{base}_S{S}"})
    run = GpuRun(wl, training=True)
    g = run.oracle_route()
    check_routing_equal(run, g)
    b = run.bufs
    assert np.allclose(f64(b["topk_w"]), g["weights"], rtol=2e-6, atol=1e-7)
    assert abs(float(b["l_aux"].item()) - g["l_aux"]) <= 1e-5 * abs(g["l_aux"])
    assert N.moe_get_device_error() == 0


def test_gate_on_two_streams_at_once():
    """Two single-launch gates in flight on different streams (each takes its
    own grid-barrier words) give the same routing as the same calls made one
    after the other; repeated calls reuse the barrier words cleanly."""
    wls = [WORKLOADS["e64_bf16"].scaled(9000), WORKLOADS["skew_e16_drop"].scaled(7000)]
    runs = [GpuRun(w) for w in wls]      # serial reference calls
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for w, r in zip(wls, runs):
        b = L.alloc_buffers(r.cfg, DEV)
        outs.append((b, L.alloc_workspace(r.cfg, DEV)))
    torch.cuda.synchronize()
    for _ in range(3):
        for (b, ws), r, st in zip(outs, runs, streams):
            d = r.d
            N.moe_gate_topk(r.cfg, d.x, d.w_gate, d.logit_bias, b["logits"], None, b["topk_idx"],
                            b["topk_w"], b["slot"], b["routed_cnt"], b["kept_cnt"],
                            b["expert_offsets"], b["row_src"], b["l_aux"], ws, st)
    torch.cuda.synchronize()
    for (b, _), r in zip(outs, runs):
        for key in ("topk_idx", "slot", "routed_cnt", "kept_cnt", "expert_offsets", "topk_w",
                    "l_aux"):
            assert torch.equal(b[key], r.bufs[key]), key
        R = r.num_rows
        assert torch.equal(b["row_src"][:R], r.bufs["row_src"][:R])
    assert N.moe_get_device_error() == 0
