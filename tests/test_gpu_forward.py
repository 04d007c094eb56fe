"""GPU forward parity of the whole layer and of each entry point.

Oracle-sized cases (same layer shape, smaller batch, nonzero biases so the
fused bias epilogue is exercised) and the layer configurations at their own
sizes both compare every element of every stage."""
import numpy as np
import pytest
import torch

from _harness import (DEV, ErrAcc, GpuRun, WORKLOADS, assert_close, check_routing_equal, f64,
                      i64, oracle_cfg)
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


@pytest.mark.parametrize("name", ["e8_bf16", "e64_bf16", "skew_e16_drop", "skew_e16_nodrop"])
def test_forward_every_element_full_size(name):
    """The layer configurations at their own sizes, every element of every
    stage against the oracle under the GPU's routing: x_disp bit for bit,
    h_pre, h and out_disp expert by expert (the oracle's expert FFN applied
    to the GPU's dispatched rows), y end to end (the oracle's out combined
    with the oracle's weights)."""
    wl = WORKLOADS[name]
    run = GpuRun(wl, training=True)
    g = run.oracle_route()
    check_routing_equal(run, g)
    rt = g["routing"]
    R = run.num_rows
    b = run.bufs
    d_model = wl.hidden_size
    # every dispatched row is an exact copy of its token (checked on the GPU)
    src = torch.as_tensor(rt.row_src // wl.k, device=DEV)
    assert torch.equal(b["x_disp"][:R], run.d.x[src])
    x_disp, h_pre, h, out = (b[n][:R].cpu() for n in ("x_disp", "h_pre", "h", "out_disp"))
    inp = run.inp
    acc = {n: ErrAcc(n) for n in ("h_pre", "h", "out_disp")}
    out_ref = np.zeros((R, d_model))
    for e in range(wl.num_experts):
        a, z = int(rt.offsets[e]), int(rt.offsets[e + 1])
        if a == z:
            continue
        hp_e, h_e, o_e = O.expert_ffn(f64(x_disp[a:z]), np.array([0, z - a]), f64(inp.w1[e:e + 1]),
                                      f64(inp.b1[e:e + 1]), f64(inp.w2[e:e + 1]),
                                      f64(inp.b2[e:e + 1]), wl.act)
        acc["h_pre"].add(f64(h_pre[a:z]), hp_e)
        acc["h"].add(f64(h[a:z]), h_e)
        acc["out_disp"].add(f64(out[a:z]), o_e)
        out_ref[a:z] = o_e
    stats = {n: a.check(wl.dtype) for n, a in acc.items()}
    y_ref = O.combine(out_ref, rt, g["weights"], d_model)
    stats["y"] = assert_close(f64(run.y), y_ref, wl.dtype, "y")
    dropped = int(np.count_nonzero((rt.slot < 0).all(axis=1)))
    print(name, f"rows={R} fully dropped tokens={dropped}", stats)


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
