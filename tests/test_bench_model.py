"""The bench's step-roofline model (CPU only): each kernel's floor is the
larger of its tensor time and its memory time, with the bytes written out
here by hand for the training layer (S=8192, d=1024, f=4096, E=32, top-2,
every choice kept: R = 16384 rows)."""
import bench
from mixture_experts_layer_86_b300.inputs import WORKLOADS

PEAKS = {"bf16_tflops": 1000.0, "hbm_gbs": 5000.0}


def test_training_step_floors():
    wl = WORKLOADS["train_e32"]
    S, d, f, E, k = 8192, 1024, 4096, 32, 2
    R = S * k
    out = bench.step_roofline(wl, R, PEAKS, ms_per_step=1.0)
    kern = out["kernels"]
    flop = 2.0 * R * d * f
    t_tc = flop / 1e15 * 1e6                         # µs at 1000 TFLOP/s
    mem = lambda nbytes: nbytes / 5e12 * 1e6         # µs at 5000 GB/s
    # weight gradients: two bf16 operands read, dW written in bf16 (the
    # layer dtype)
    dw_bytes = R * d * 2 + R * f * 2 + E * d * f * 2
    assert kern["dW2"]["bytes"] == dw_bytes == kern["dW1"]["bytes"]
    assert kern["dW1"]["bound"] == "tensor"
    assert abs(kern["dW1"]["us"] - round(max(t_tc, mem(dw_bytes)), 2)) < 1e-9
    # W1 in training writes h_pre and h
    w1_bytes = E * f * d * 2 + R * d * 2 + 2 * R * f * 2
    assert kern["W1"]["bytes"] == w1_bytes
    assert abs(kern["W1"]["us"] - round(max(t_tc, mem(w1_bytes)), 2)) < 1e-9
    # dh reads W2, dO and h_pre, writes dh_pre; dx_disp reads W1 and dh_pre
    assert kern["dh"]["bytes"] == E * d * f * 2 + R * d * 2 + 2 * R * f * 2
    assert kern["dx_disp"]["bytes"] == E * f * d * 2 + R * f * 2 + R * d * 2
    assert kern["W2"]["flop"] == flop and kern["dx_disp"]["flop"] == flop
    # the floor is the sum of the per-kernel floors; frac = floor / step
    total_us = sum(v["us"] for v in kern.values())
    assert abs(out["floor_ms"] - total_us * 1e-3) < 1e-12
    assert abs(out["frac"] - out["floor_ms"] / 1.0) < 1e-12


def test_forward_only_floor_has_no_backward_kernels():
    wl = WORKLOADS["e64_bf16"]
    R = 32762
    out = bench.step_roofline(wl, R, PEAKS, ms_per_step=2.0)
    assert set(out["kernels"]) == {"gate", "dispatch", "W1", "W2", "combine"}
    # inference W1 writes h only
    S, d, f, E = 16384, 2048, 5120, 64
    assert out["kernels"]["W1"]["bytes"] == E * f * d * 2 + R * d * 2 + R * f * 2
    assert out["kernels"]["W1"]["bound"] == "tensor"
