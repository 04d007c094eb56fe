"""GPU forward parity of the whole layer and of each entry point.

Oracle-sized cases (same layer shape, smaller batch, nonzero biases so the
fused bias epilogue is exercised) compare every element; full-size cases
compare the dispatch copy exactly and y on sampled tokens."""
import numpy as np
import pytest
import torch

from _harness import (DEV, GpuRun, WORKLOADS, assert_close, check_routing_equal, f64, i64,
                      oracle_cfg, oracle_token_outputs)
from mixture_experts_layer_86_b300 import _native as N
from mixture_experts_layer_86_b300 import layer as L
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

SMALL = [("tiny_fp32", 256), ("e8_bf16", 1000), ("e64_bf16", 300), ("skew_e16_drop", 700),
         ("skew_e16_nodrop", 700), ("train_e32", 600), ("decode_e64", 256)]


def _small(name, S):
    return WORKLOADS[name].scaled(S, bias_std=0.1)


@pytest.mark.parametrize("name,S", SMALL)
def test_forward_parity_elementwise(name, S):
    wl = _small(name, S)
    run = GpuRun(wl, training=True)
    g = run.oracle_route()
    check_routing_equal(run, g)
    inp = run.inp
    ref = O.forward(oracle_cfg(wl), f64(inp.x), None, f64(inp.w1), f64(inp.b1), f64(inp.w2),
                    f64(inp.b2), logits=f64(run.bufs["logits"]))
    R = run.num_rows
    assert R == ref["routing"].num_rows
    b = run.bufs
    # dispatch is a copy: bit-exact
    assert np.array_equal(f64(b["x_disp"][:R]), ref["x_disp"])
    # each stage against the oracle applied to the GPU's own stage input
    h_pre_ref, h_ref, out_ref = O.expert_ffn(f64(b["x_disp"][:R]), ref["routing"].offsets,
                                             f64(inp.w1), f64(inp.b1), f64(inp.w2), f64(inp.b2),
                                             wl.act)
    assert_close(f64(b["h_pre"][:R]), h_pre_ref, wl.dtype, "h_pre")
    assert_close(f64(b["h"][:R]), h_ref, wl.dtype, "h")
    assert_close(f64(b["out_disp"][:R]), out_ref, wl.dtype, "out_disp")
    y_from_out = O.combine(f64(b["out_disp"][:R]), ref["routing"], ref["weights"], wl.hidden_size)
    assert_close(f64(run.y), y_from_out, wl.dtype, "combine")
    # end to end
    stats = assert_close(f64(run.y), ref["y"], wl.dtype, "y")
    assert abs(float(run.l_aux.item()) - ref["l_aux"]) <= 1e-5 * abs(ref["l_aux"])
    assert np.array_equal(i64(run.kept), ref["routing"].kept)
    print(name, S, stats)


@pytest.mark.parametrize("name", ["e8_bf16", "e64_bf16", "skew_e16_drop", "skew_e16_nodrop",
                                  "train_e32"])
def test_forward_full_size_sampled(name):
    wl = WORKLOADS[name]
    run = GpuRun(wl)
    g = run.oracle_route()
    check_routing_equal(run, g)
    rt = g["routing"]
    R = run.num_rows
    b = run.bufs
    # every dispatched row is an exact copy of its token (checked on the GPU)
    src = torch.as_tensor(rt.row_src // wl.k, device=DEV)
    assert torch.equal(b["x_disp"][:R], run.d.x[src])
    # y on sampled tokens (first, last, random, and some with dropped choices)
    gen = np.random.default_rng(7)
    S = wl.num_tokens
    toks = set([0, 1, S - 1]) | set(gen.choice(S, 40, replace=False).tolist())
    dropped = np.nonzero((rt.slot < 0).any(axis=1))[0]
    toks |= set(dropped[:8].tolist())
    toks = sorted(toks)
    ref = oracle_token_outputs(run, g, toks)
    stats = assert_close(f64(run.y[toks]), ref, wl.dtype, "y sampled")
    print(name, "dropped tokens:", len(dropped), stats)


def test_entry_points_compose_to_forward():
    """moe_gate_topk -> moe_dispatch -> moe_expert_ffn -> moe_combine gives
    moe_forward's output bit for bit."""
    wl = _small("e8_bf16", 777)
    run = GpuRun(wl)
    cfg, d = run.cfg, run.d
    bufs = L.alloc_buffers(cfg, DEV)
    ws = L.alloc_workspace(cfg, DEV)
    N.moe_gate_topk(cfg, d.x, d.w_gate, d.logit_bias, bufs["logits"], None, bufs["topk_idx"],
                    bufs["topk_w"], bufs["slot"], bufs["routed_cnt"], bufs["kept_cnt"],
                    bufs["expert_offsets"], bufs["row_src"], bufs["l_aux"], ws)
    N.moe_dispatch(cfg, d.x, bufs["topk_idx"], bufs["slot"], bufs["expert_offsets"], bufs["x_disp"])
    N.moe_expert_ffn(cfg, bufs["x_disp"], bufs["expert_offsets"], d.w1, d.b1, d.w2, d.b2, None,
                     bufs["h"], bufs["out_disp"])
    y = torch.empty_like(d.x)
    N.moe_combine(cfg, bufs["out_disp"], bufs["topk_idx"], bufs["slot"], bufs["expert_offsets"],
                  bufs["topk_w"], y)
    torch.cuda.synchronize()
    assert torch.equal(y, run.y)
    assert torch.equal(bufs["l_aux"], run.l_aux)
    assert N.moe_get_device_error() == 0
