"""GPU backward parity: gradients of <dY, y> + aux_loss_weight * l_aux with
respect to x, W_g, W1, b1, W2, b2, against the oracle's backward under the
GPU's routing.  Includes an expert that receives no token (its weight
gradients must be written as exact zeros)."""
import numpy as np
import pytest
import torch

from _harness import DEV, GpuRun, WORKLOADS, assert_close, check_routing_equal, f64, oracle_cfg
from mixture_experts_layer_86_b300 import _native as N
from mixture_experts_layer_86_b300.inputs import Workload, make_inputs
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu


def _oracle_grads(run):
    wl, inp = run.wl, run.inp
    lb = None if inp.logit_bias is None else f64(inp.logit_bias)
    ref = O.forward(oracle_cfg(wl), f64(inp.x), f64(inp.w_gate), f64(inp.w1), f64(inp.b1),
                    f64(inp.w2), f64(inp.b2), logit_bias=lb, logits=f64(run.bufs["logits"]))
    return ref, O.backward(oracle_cfg(wl), ref, f64(inp.x), f64(inp.w_gate), f64(inp.w1),
                           f64(inp.w2), f64(inp.dy))


def _check_all(run, ref, gref):
    g = run.grads
    dt = run.wl.dtype
    out = {}
    for key in ("dx", "dw_gate", "dw1", "db1", "dw2", "db2"):
        out[key] = assert_close(f64(g[key]), gref[key], dt, key)
    return out


@pytest.mark.parametrize("name,S", [("train_e32", 600), ("train_e32", 1500), ("e8_bf16", 900),
                                    ("tiny_fp32", 256)])
def test_backward_parity(name, S):
    wl = WORKLOADS[name].scaled(S, bias_std=0.1, backward=True,
                                aux_loss_weight=WORKLOADS[name].aux_loss_weight or 0.01)
    run = GpuRun(wl, training=True)
    run.backward()
    ref, gref = _oracle_grads(run)
    check_routing_equal(run, ref)
    print(name, S, _check_all(run, ref, gref))


def test_backward_odd_widths():
    """d = 96 and f = 160 are multiples of 8 but not of the 64-wide TMA boxes
    or the 256-wide weight-gradient tiles: partial boxes on both sides and
    bias-gradient columns past the end of the tile."""
    wl = Workload("odd_widths", 700, 96, 160, 6, 2, 1.25, 4, True, "gelu_tanh", "bf16",
                  seed=13, bias_std=0.1, aux_loss_weight=0.01, backward=True)
    run = GpuRun(wl, training=True)
    run.backward()
    ref, gref = _oracle_grads(run)
    check_routing_equal(run, ref)
    print("odd widths", _check_all(run, ref, gref))


@pytest.mark.parametrize("S,d,f,E,k", [(1200, 128, 64, 256, 2), (900, 2048, 256, 64, 2),
                                        (333, 512, 128, 8, 1), (5, 64, 64, 4, 2)])
def test_backward_router_shapes(S, d, f, E, k):
    """The router's tensor-core backward (dW_g over token chunks, dX with the
    experts' rows added in the GEMM epilogue) at expert counts whose [hi | lo]
    operand spans one to eight 64-wide blocks, hidden sizes of one to sixteen
    128-column tiles, and a batch smaller than one 64-row K block."""
    wl = Workload(f"router_e{E}", S, d, f, E, k, 1.25, 4, True, "gelu_tanh", "bf16", seed=21,
                  bias_std=0.1, aux_loss_weight=0.01, backward=True)
    run = GpuRun(wl, training=True)
    run.backward()
    assert N.moe_get_device_error() == 0
    ref, gref = _oracle_grads(run)
    check_routing_equal(run, ref)
    print("router shapes", S, d, E, {k_: f"{v['rel_l2']:.2e}" for k_, v in _check_all(run, ref, gref).items()})


def test_backward_empty_expert_gets_zero_gradient():
    wl = WORKLOADS["train_e32"].scaled(400, bias_std=0.1, backward=True, skew=0.0)
    inp = make_inputs(wl)
    # expert 5 can never win: a large negative logit bias
    bias = torch.zeros(wl.num_experts)
    bias[5] = -1e4
    inp.logit_bias = bias
    run = GpuRun(wl, training=True, inp=inp)
    # poison the gradient buffers so "not written" cannot pass as zero
    grads = {k: torch.full(s, float("nan"), dtype=torch.bfloat16, device=DEV) for k, s in (
        ("dx", run.d.x.shape), ("dw_gate", run.d.w_gate.shape), ("dw1", run.d.w1.shape),
        ("db1", run.d.w1.shape[:2]), ("dw2", run.d.w2.shape), ("db2", run.d.w2.shape[:2]))}
    from mixture_experts_layer_86_b300 import layer as L
    run.grads = L.backward(run.cfg, run.d.x, run.d.w_gate, run.d.w1, run.d.w2, run.bufs,
                           run.d.dy, grads=grads)
    torch.cuda.synchronize()
    assert int(run.kept[5].item()) == 0
    for key in ("dw1", "db1", "dw2", "db2"):
        assert torch.all(run.grads[key][5] == 0), key
    ref, gref = _oracle_grads(run)
    _check_all(run, ref, gref)


def test_training_step_every_element_full_size():
    """The training configuration at its own size (S=8192, d=1024, E=32,
    f=4096, ~512 rows per expert): the forward stages and all six gradients,
    every element, against the oracle's forward and backward under the GPU's
    routing.  At this size the weight-gradient GEMM runs 8 K blocks per tile
    and the data-gradient GEMM two 256-token tiles per expert."""
    wl = WORKLOADS["train_e32"]
    run = GpuRun(wl, training=True)
    run.backward()
    assert N.moe_get_device_error() == 0
    ref, gref = _oracle_grads(run)
    check_routing_equal(run, ref)
    R = run.num_rows
    b = run.bufs
    stats = {}
    assert np.array_equal(f64(b["x_disp"][:R]), ref["x_disp"])
    for key, name in (("h_pre", "h_pre"), ("h", "h"), ("out", "out_disp")):
        stats[name] = assert_close(f64(b[name][:R]), ref[key], wl.dtype, name)
    stats["y"] = assert_close(f64(run.y), ref["y"], wl.dtype, "y")
    stats.update(_check_all(run, ref, gref))
    print("train_e32 full size", {k: f"{v['rel_l2']:.2e}" for k, v in stats.items()})
