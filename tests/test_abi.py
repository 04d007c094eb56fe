"""The C-ABI library loads, exports every symbol the header declares, and its
host-side logic (capacity arithmetic, buffer sizing, argument checks) is
right.  No call here reaches a GPU: every device entry point is called only
with arguments its host-side checks reject before anything is enqueued."""
import ctypes
import os
import random
import re

import pytest

from mixture_experts_layer_86_b300 import _native as N
from oracle import moe_oracle as O

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "moe_b300.h")


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|moe_status|int64_t)\s*(moe_\w+)\s*\(",
                                 src, re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("moe_gate_topk", "moe_dispatch", "moe_expert_ffn", "moe_combine",
                     "moe_forward", "moe_backward"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = N.library()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(N.exported_symbols())


def test_status_strings():
    assert N.status_string(N.MOE_OK) == "MOE_OK"
    assert N.status_string(N.MOE_ERR_WORKSPACE) == "MOE_ERR_WORKSPACE"
    assert N.status_string(99) == "MOE_ERR_UNKNOWN"


def test_capacity_matches_oracle():
    rng = random.Random(0)
    cfs = ["0.25", "0.5", "1.0", "1.1", "1.2", "1.25", "1.5", "2.0", "0.3", "3.7", "1.000001"]
    for _ in range(2000):
        S = rng.choice([0, 1, 7, 100, 256, 4096, 16384, rng.randrange(1, 1 << 20)])
        E = rng.randrange(2, 257)
        k = rng.choice([1, 2])
        cf = rng.choice(cfs)
        mc = rng.randrange(0, 9)
        drop = rng.random() < 0.8
        cfg = N.make_config(S, 64, 64, E, k, float(cf), mc, drop)
        want = O.capacity(S, E, k, cf, mc, drop)
        got = N.moe_capacity(cfg)
        assert got == (-1 if want is None else want), (S, E, k, cf, mc, drop)
        rows = N.moe_max_rows(cfg)
        assert rows == (S * k if want is None else min(S * k, E * want))


def test_layer_config_capacities():
    from mixture_experts_layer_86_b300.inputs import WORKLOADS
    want = {"tiny_fp32": 64, "e8_bf16": 1024, "e64_bf16": 640, "skew_e16_drop": 2048,
            "skew_e16_nodrop": -1, "train_e32": 640,
            "decode_e64": 8}  # max(4, ceil(256*2*1.0/64))
    for name, wl in WORKLOADS.items():
        assert N.moe_capacity(N.config_from_workload(wl)) == want[name]


def test_workspace_sizes():
    cfg = N.make_config(16384, 2048, 5120, 64, 2, 1.25, 4, True)
    fwd, bwd = N.moe_workspace_size(cfg), N.moe_workspace_size(cfg, True)
    assert fwd >= 16384 * 64 * 4 and bwd > fwd
    small = N.make_config(0, 8, 8, 2, 1, 1.0, 0, True)
    assert N.moe_workspace_size(small) >= 0


@pytest.mark.parametrize("bad,status", [
    (dict(k=3), N.MOE_ERR_INVALID_ARG), (dict(k=0), N.MOE_ERR_INVALID_ARG),
    (dict(num_experts=1, k=2), N.MOE_ERR_INVALID_ARG),
    (dict(hidden_size=36), N.MOE_ERR_INVALID_ARG), (dict(ffn_size=4), N.MOE_ERR_INVALID_ARG),
    (dict(capacity_factor=0.0), N.MOE_ERR_INVALID_ARG),
    (dict(capacity_factor=-1.0), N.MOE_ERR_INVALID_ARG),
    (dict(min_capacity=-1), N.MOE_ERR_INVALID_ARG), (dict(num_tokens=-5), N.MOE_ERR_INVALID_ARG),
    (dict(act=7), N.MOE_ERR_INVALID_ARG), (dict(dtype=5), N.MOE_ERR_INVALID_ARG),
    (dict(num_experts=300), N.MOE_ERR_UNSUPPORTED),
    (dict(num_tokens=1 << 30, k=2), N.MOE_ERR_UNSUPPORTED),
])
def test_invalid_configs_rejected(bad, status):
    base = dict(num_tokens=64, hidden_size=32, ffn_size=64, num_experts=4, k=1,
                capacity_factor=1.0, min_capacity=4, drop_tokens=True)
    base.update({k: v for k, v in bad.items() if k not in ("act", "dtype")})
    cfg = N.make_config(**base, act=bad.get("act", "relu"), dtype=bad.get("dtype", "f32"))
    v = ctypes.c_int64()
    assert N.library().moe_capacity(ctypes.byref(cfg), ctypes.byref(v)) == status


FAKE = 0x7f0000000000          # aligned, never dereferenced: checks fail first
MISALIGNED = FAKE + 8


def _gate_args(cfg, **over):
    names = ["x", "w_gate", "logit_bias", "logits", "probs", "topk_idx", "topk_w", "slot",
             "routed_cnt", "kept_cnt", "expert_offsets", "row_src", "l_aux", "workspace"]
    vals = {n: FAKE for n in names}
    vals.update(logit_bias=None, logits=None, probs=None)
    vals.update(over)
    ws = over.get("ws_bytes", 1 << 40)
    return [ctypes.byref(cfg)] + [vals[n] for n in names] + [ws, None]


def test_null_misaligned_and_workspace_checks():
    lib = N.library()
    cfg = N.make_config(64, 32, 64, 4, 1, 1.0, 4, True, "relu", "f32")
    assert lib.moe_gate_topk(*_gate_args(cfg, x=None)) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_gate_topk(*_gate_args(cfg, slot=None)) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_gate_topk(*_gate_args(cfg, x=MISALIGNED)) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_gate_topk(*_gate_args(cfg, probs=MISALIGNED)) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_gate_topk(*_gate_args(cfg, ws_bytes=16)) == N.MOE_ERR_WORKSPACE
    assert lib.moe_dispatch(ctypes.byref(cfg), FAKE, FAKE, None, FAKE, FAKE, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(ctypes.byref(cfg), FAKE, FAKE, FAKE, FAKE, FAKE, MISALIGNED, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_expert_ffn(ctypes.byref(cfg), FAKE, FAKE, FAKE, None, FAKE, FAKE, None, FAKE, FAKE,
                              None) == N.MOE_ERR_INVALID_ARG
    bufs = N.MoeBuffers()
    assert lib.moe_forward(ctypes.byref(cfg), FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE,
                           ctypes.byref(bufs), FAKE, 1 << 40, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_backward(ctypes.byref(cfg), FAKE, FAKE, FAKE, FAKE, ctypes.byref(bufs), FAKE,
                            FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == N.MOE_ERR_INVALID_ARG
    full = N.MoeBuffers(*([FAKE] * 14))
    assert lib.moe_backward(ctypes.byref(cfg), FAKE, FAKE, FAKE, FAKE, ctypes.byref(full), FAKE,
                            FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, None) == N.MOE_ERR_WORKSPACE
    bad = N.make_config(64, 32, 64, 4, 3, 1.0, 4, True)
    assert lib.moe_gate_topk(*_gate_args(bad)) == N.MOE_ERR_INVALID_ARG


def test_residual_mix_argument_checks():
    """moe_forward_residual takes the learned mix's three arguments all
    together or none of them; the checks run before anything is enqueued."""
    lib = N.library()
    cfg = N.make_config(64, 32, 64, 4, 1, 1.0, 4, True, "relu", "f32")
    full = N.MoeBuffers(*([FAKE] * 14))

    def call(mix_w, mix_b, mix):
        return lib.moe_forward_residual(ctypes.byref(cfg), FAKE, FAKE, None, FAKE, FAKE, FAKE,
                                        FAKE, FAKE, FAKE, FAKE, FAKE, mix_w, mix_b, mix, FAKE,
                                        ctypes.byref(full), FAKE, FAKE, FAKE, 1 << 40, None)

    assert call(FAKE, FAKE, None) == N.MOE_ERR_INVALID_ARG
    assert call(FAKE, None, FAKE) == N.MOE_ERR_INVALID_ARG
    assert call(None, FAKE, None) == N.MOE_ERR_INVALID_ARG
    assert call(None, None, FAKE) == N.MOE_ERR_INVALID_ARG
    assert call(MISALIGNED, FAKE, FAKE) == N.MOE_ERR_INVALID_ARG
    assert call(FAKE, FAKE, MISALIGNED) == N.MOE_ERR_INVALID_ARG


def test_fused_dispatch_argument_checks():
    """moe_expert_ffn_gather checks every pointer on the host and refuses fp32
    layers (the gather form is a tensor-core GEMM); moe_forward without an
    x_disp buffer is refused for an fp32 layer.  Nothing is enqueued."""
    lib = N.library()
    f32 = N.make_config(64, 32, 64, 4, 1, 1.0, 4, True, "relu", "f32")
    bf = N.make_config(64, 32, 64, 4, 1, 1.0, 4, True, "relu", "bf16")

    def gather(cfg, **o):
        names = ("x", "row_src", "offsets", "w1", "b1", "w2", "b2")
        return lib.moe_expert_ffn_gather(ctypes.byref(cfg), *[o.get(n, FAKE) for n in names],
                                         o.get("h_pre"), o.get("h", FAKE), o.get("out", FAKE),
                                         None)

    assert gather(f32) == N.MOE_ERR_UNSUPPORTED
    assert gather(bf, row_src=None) == N.MOE_ERR_INVALID_ARG
    assert gather(bf, x=MISALIGNED) == N.MOE_ERR_INVALID_ARG
    assert gather(bf, h_pre=MISALIGNED) == N.MOE_ERR_INVALID_ARG
    assert gather(bf, out=None) == N.MOE_ERR_INVALID_ARG
    nodisp = N.MoeBuffers(*([FAKE] * 14))
    nodisp.x_disp = None
    assert lib.moe_forward(ctypes.byref(f32), FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE,
                           ctypes.byref(nodisp), FAKE, 1 << 40, None) == N.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("bad", [dict(noise_policy=3), dict(noise_policy=-1),
                                 dict(second_expert_sampling=2), dict(use_rts=5),
                                 dict(jitter_eps=-0.1), dict(jitter_eps=1.0)])
def test_invalid_noise_options_rejected(bad):
    cfg = N.make_config(64, 32, 64, 4, 2, 1.0, 4, True, "relu", "f32")
    for k, v in bad.items():
        setattr(cfg, k, v)
    rows = ctypes.c_int64()
    assert N.library().moe_max_rows(ctypes.byref(cfg), ctypes.byref(rows)) == N.MOE_ERR_INVALID_ARG


def test_noise_workspace_holds_the_jittered_input():
    base = N.make_config(4096, 512, 64, 8, 2, 1.0, 4, True)
    jit = N.make_config(4096, 512, 64, 8, 2, 1.0, 4, True, noise_policy="jitter")
    extra = N.moe_workspace_size(jit) - N.moe_workspace_size(base)
    assert extra >= 4096 * 512 * 2
    assert N.moe_workspace_size(jit, True) - N.moe_workspace_size(base, True) >= 4096 * 512 * 2
