"""GPU parity of the gating variants (readings R9 and R10 of the oracle):
the gate temperature T (p = softmax(logits / T)), the std-based balance loss
lambda * (std_e(mean_s p[s,e]) + 1e-6), and noisy gating as caller-drawn
per-token logit noise [S, E].  Routing must be bit-exact against the oracle
fed the GPU's own logits; probabilities, weights, l_aux, y and every
gradient within the layer's tolerances."""
import dataclasses

import numpy as np
import pytest

from _harness import GpuRun, WORKLOADS, assert_close, check_routing_equal, f64, oracle_cfg
from mixture_experts_layer_86_b300 import _native as N
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

VARIANTS = {
    "temp0.5": dict(gate_temperature=0.5),
    "temp2_std": dict(gate_temperature=2.0, aux_loss_type="std"),
    "noise_std": dict(logit_noise_std=0.5, aux_loss_type="std"),
    "noise_temp0.5": dict(logit_noise_std=0.3, gate_temperature=0.5),
}


def _wl(name, S, variant, backward=False):
    wl = WORKLOADS[name].scaled(S, bias_std=0.1)
    extra = dict(VARIANTS[variant])
    if backward:
        extra.update(backward=True, aux_loss_weight=0.05)
    return dataclasses.replace(wl, name=f"{wl.name}+{variant}", **extra)


def _oracle(run):
    inp = run.inp
    lb = None if inp.logit_bias is None else f64(inp.logit_bias)
    return O.forward(oracle_cfg(run.wl), f64(inp.x), f64(inp.w_gate), f64(inp.w1), f64(inp.b1),
                     f64(inp.w2), f64(inp.b2), logit_bias=lb, logits=f64(run.bufs["logits"]))


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("name,S", [("tiny_fp32", 256), ("e8_bf16", 900), ("skew_e16_drop", 600)])
def test_gating_variant_forward(name, S, variant):
    run = GpuRun(_wl(name, S, variant), training=True)
    ref = _oracle(run)
    check_routing_equal(run, ref)
    b = run.bufs
    # the stored logits include the bias / noise, before the 1/T scaling
    inp = run.inp
    lg = O.gate_logits(f64(inp.x), f64(inp.w_gate),
                       None if inp.logit_bias is None else f64(inp.logit_bias))
    assert np.abs(f64(b["logits"]) - lg).max() <= 1e-5 * np.abs(lg).max()
    assert np.allclose(f64(b["probs"]), ref["probs"], rtol=2e-6, atol=1e-7)
    assert np.allclose(f64(b["topk_w"]), ref["weights"], rtol=2e-6, atol=1e-7)
    assert abs(float(run.l_aux.item()) - ref["l_aux"]) <= 1e-5 * abs(ref["l_aux"]) + 1e-9
    assert_close(f64(run.y), ref["y"], run.wl.dtype, "y")
    assert N.moe_get_device_error() == 0


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("name,S", [("tiny_fp32", 256), ("train_e32", 700)])
def test_gating_variant_backward(name, S, variant):
    run = GpuRun(_wl(name, S, variant, backward=True), training=True)
    run.backward()
    ref = _oracle(run)
    check_routing_equal(run, ref)
    inp = run.inp
    gref = O.backward(oracle_cfg(run.wl), ref, f64(inp.x), f64(inp.w_gate), f64(inp.w1),
                      f64(inp.w2), f64(inp.dy))
    for key in ("dx", "dw_gate", "dw1", "db1", "dw2", "db2"):
        assert_close(f64(run.grads[key]), gref[key], run.wl.dtype, key)
    assert N.moe_get_device_error() == 0
