"""moe_gate_topk_static -- the gate entry point for callers that cannot
allocate device memory (they hold only their input / output buffers and a
stream, so they cannot hand moe_gate_topk its workspace).  It must give the
same results as moe_gate_topk, call after call, with its scratch compiled
into the library.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_86_b300 import _native as N
from mixture_experts_layer_86_b300 import layer as L
from mixture_experts_layer_86_b300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _outputs(cfg, sentinel):
    S, E, k = cfg.num_tokens, cfg.num_experts, cfg.k
    R = max(N.moe_max_rows(cfg), 1)
    i32 = dict(dtype=torch.int32, device=DEV)
    f32 = dict(dtype=torch.float32, device=DEV)
    return {"logits": torch.full((S, E), sentinel, **f32),
            "probs": torch.full((S, E), sentinel, **f32),
            "topk_idx": torch.full((S, k), -9, **i32),
            "topk_w": torch.full((S, k), sentinel, **f32),
            "slot": torch.full((S, k), -9, **i32),
            "routed_cnt": torch.full((E,), -9, **i32), "kept_cnt": torch.full((E,), -9, **i32),
            "expert_offsets": torch.full((E + 1,), -9, **i32),
            "row_src": torch.full((R,), -9, **i32), "l_aux": torch.full((1,), sentinel, **f32)}


def _call(fn, cfg, inp, o, logits=True, *extra):
    return fn(cfg, inp.x, inp.w_gate, inp.logit_bias, o["logits"] if logits else None, o["probs"],
              o["topk_idx"], o["topk_w"], o["slot"], o["routed_cnt"], o["kept_cnt"],
              o["expert_offsets"], o["row_src"], o["l_aux"], *extra)


def _same(ref, got, with_logits=True):
    R = int(ref["expert_offsets"][-1])
    for key in ("topk_idx", "slot", "routed_cnt", "kept_cnt", "expert_offsets"):
        assert torch.equal(ref[key], got[key]), key
    assert torch.equal(ref["row_src"][:R], got["row_src"][:R])
    keys = ("probs", "topk_w", "l_aux") + (("logits",) if with_logits else ())
    for key in keys:
        a, b = ref[key].double().cpu().numpy(), got[key].double().cpu().numpy()
        assert np.allclose(b, a, rtol=2e-6, atol=1e-7), key


@pytest.mark.parametrize("wl", [
    Workload("gate_e8", 1000, 512, 64, 8, 2, 1.0, 4, True, "gelu_tanh", "bf16", seed=1),
    Workload("gate_e64", 16384, 2048, 64, 64, 2, 1.25, 4, True, "gelu_tanh", "bf16", seed=2),
    Workload("gate_skew", 3000, 1024, 64, 16, 2, 2.0, 4, False, "gelu_tanh", "bf16", seed=3,
             skew=1.2),
    Workload("gate_f32", 256, 32, 64, 4, 1, 1.0, 4, True, "relu", "f32", seed=0),
], ids=lambda w: w.name)
def test_static_gate_matches_workspace_gate_twice(wl):
    cfg = N.config_from_workload(wl)
    inp = make_inputs(wl).to(DEV)
    ref = _outputs(cfg, 0.0)
    ws = L.alloc_workspace(cfg, DEV)
    _call(N.moe_gate_topk, cfg, inp, ref, True, ws)
    torch.cuda.synchronize()
    for sentinel in (float("nan"), -3.0):   # two calls in a row, different stale outputs
        got = _outputs(cfg, sentinel)
        _call(N.moe_gate_topk_static, cfg, inp, got, True)
        torch.cuda.synchronize()
        _same(ref, got)
    assert N.moe_get_device_error() == 0


def test_static_gate_fp32_uses_builtin_logits_scratch():
    wl = Workload("gate_f32_nolog", 2000, 64, 64, 8, 2, 1.25, 4, True, "relu", "f32", seed=4)
    cfg = N.config_from_workload(wl)
    inp = make_inputs(wl).to(DEV)
    ref = _outputs(cfg, 0.0)
    _call(N.moe_gate_topk, cfg, inp, ref, False, L.alloc_workspace(cfg, DEV))
    for _ in range(2):
        got = _outputs(cfg, float("nan"))
        _call(N.moe_gate_topk_static, cfg, inp, got, False)
        torch.cuda.synchronize()
        _same(ref, got, with_logits=False)


def test_static_gate_allocates_no_device_memory():
    """After the first call on the device (which looks up the scratch
    array's address), further calls leave both torch's allocator and the
    device's free memory exactly as they were."""
    wl = Workload("gate_e64_mem", 4096, 2048, 64, 64, 2, 1.25, 4, True, "gelu_tanh", "bf16",
                  seed=2)
    cfg = N.config_from_workload(wl)
    inp = make_inputs(wl).to(DEV)
    got = _outputs(cfg, 0.0)
    _call(N.moe_gate_topk_static, cfg, inp, got, True)
    torch.cuda.synchronize()
    allocated0 = torch.cuda.memory_allocated()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        _call(N.moe_gate_topk_static, cfg, inp, got, True)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == allocated0
    assert free1 == free0, (free0, free1)
    assert N.moe_get_device_error() == 0


def test_static_gate_rejects_configs_beyond_its_scratch():
    cfg = N.make_config(1 << 20, 64, 64, 64, 2, 1.0, 4, True)   # S*E*4 = 256 MiB of logits
    fake = 1 << 44
    st = N.library().moe_gate_topk_static(
        cfg, fake, fake, None, None, None, fake, fake, fake, fake, fake, fake, fake, fake, None)
    assert st == N.MOE_ERR_WORKSPACE
