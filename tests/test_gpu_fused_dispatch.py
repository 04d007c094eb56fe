"""The dispatch fused into the first expert GEMM (moe_expert_ffn_gather, and
moe_forward without an x_disp buffer): the GEMM reads each expert's token
rows straight from x, so h_pre, h, out_disp and y must equal the dispatch +
grouped FFN path bit for bit, and through it the oracle."""
import numpy as np
import pytest
import torch

from _harness import DEV, GpuRun, WORKLOADS, assert_close, check_routing_equal, f64, oracle_cfg
from mixture_experts_layer_86_b300 import _native as N
from mixture_experts_layer_86_b300 import layer as L
from mixture_experts_layer_86_b300.inputs import Workload, make_inputs
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

CASES = [
    WORKLOADS["e8_bf16"].scaled(1000, bias_std=0.1),
    WORKLOADS["e64_bf16"].scaled(300, bias_std=0.1),
    WORKLOADS["skew_e16_nodrop"].scaled(700, bias_std=0.1),
    WORKLOADS["decode_e64"],
    Workload("ragged_widths", 1001, 96, 160, 5, 1, 1.1, 3, True, "gelu_erf", "bf16", seed=21,
             bias_std=0.1),
    Workload("one_token", 1, 64, 128, 2, 2, 1.0, 1, True, "gelu_tanh", "bf16", seed=3),
    WORKLOADS["e64_bf16"],
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_gather_ffn_equals_dispatch_then_ffn(wl):
    run = GpuRun(wl, training=True)       # dispatch path, keeps x_disp and h_pre
    b, d = run.bufs, run.d
    R = max(N.moe_max_rows(run.cfg), 1)
    dt = d.x.dtype
    h_pre = torch.full((R, wl.ffn_size), float("nan"), dtype=dt, device=DEV)
    h = torch.full_like(h_pre, float("nan"))
    out = torch.full((R, wl.hidden_size), float("nan"), dtype=dt, device=DEV)
    N.moe_expert_ffn_gather(run.cfg, d.x, b["row_src"], b["expert_offsets"], d.w1, d.b1, d.w2,
                            d.b2, h_pre, h, out)
    torch.cuda.synchronize()
    rows = run.num_rows
    assert torch.equal(h_pre[:rows], b["h_pre"][:rows])
    assert torch.equal(h[:rows], b["h"][:rows])
    assert torch.equal(out[:rows], b["out_disp"][:rows])
    assert N.moe_get_device_error() == 0


@pytest.mark.parametrize("wl", CASES[:5], ids=lambda w: w.name)
def test_forward_without_x_disp_is_bit_identical(wl):
    run = GpuRun(wl)
    cfg, d = run.cfg, run.d
    bufs = L.alloc_buffers(cfg, DEV, fused_dispatch=True)
    assert bufs["x_disp"] is None
    y = torch.empty_like(d.x)
    N.moe_forward(cfg, d.x, d.w_gate, d.logit_bias, d.w1, d.b1, d.w2, d.b2, y, bufs,
                  L.alloc_workspace(cfg, DEV))
    torch.cuda.synchronize()
    assert torch.equal(y, run.y)
    assert torch.equal(bufs["l_aux"], run.l_aux)
    assert torch.equal(bufs["kept_cnt"], run.kept)
    # and so against the oracle, under the GPU's routing
    g = run.oracle_route()
    check_routing_equal(run, g)
    inp = run.inp
    ref = O.forward(oracle_cfg(wl), f64(inp.x), None, f64(inp.w1), f64(inp.b1), f64(inp.w2),
                    f64(inp.b2), logits=f64(run.bufs["logits"]))
    assert_close(f64(y), ref["y"], wl.dtype, "y")
    assert N.moe_get_device_error() == 0


def test_fused_forward_full_size_64_experts():
    """The 64-expert layer at its own size through moe_forward without
    x_disp: y bit-identical to the dispatch path."""
    wl = WORKLOADS["e64_bf16"]
    inp = make_inputs(wl).to(DEV)
    cfg = N.config_from_workload(wl)
    ys = []
    for fused in (False, True):
        y, l_aux, kept, _ = L.forward(cfg, inp.x, inp.w_gate, inp.logit_bias, inp.w1, inp.b1,
                                      inp.w2, inp.b2, fused_dispatch=fused)
        torch.cuda.synchronize()
        ys.append((y, l_aux.clone(), kept.clone()))
    assert torch.equal(ys[0][0], ys[1][0])
    assert torch.equal(ys[0][1], ys[1][1]) and torch.equal(ys[0][2], ys[1][2])
    assert N.moe_get_device_error() == 0


def test_fused_dispatch_is_bf16_only():
    wl = WORKLOADS["tiny_fp32"]
    cfg = N.config_from_workload(wl)
    inp = make_inputs(wl).to(DEV)
    bufs = L.alloc_buffers(cfg, DEV)
    with pytest.raises(N.MoeError) as ei:
        N.moe_expert_ffn_gather(cfg, inp.x, bufs["row_src"], bufs["expert_offsets"], inp.w1,
                                inp.b1, inp.w2, inp.b2, None, bufs["h"], bufs["out_disp"])
    assert ei.value.status == N.MOE_ERR_UNSUPPORTED
    bufs["x_disp"] = None
    with pytest.raises(N.MoeError) as ei:
        N.moe_forward(cfg, inp.x, inp.w_gate, None, inp.w1, inp.b1, inp.w2, inp.b2,
                      torch.empty_like(inp.x), bufs, L.alloc_workspace(cfg, DEV))
    assert ei.value.status == N.MOE_ERR_INVALID_ARG
