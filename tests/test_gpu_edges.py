"""Degenerate and boundary cases of the CUDA path: an empty batch, one
token, every token preferring one expert, no capacity cap with heavy skew,
a single expert, the largest expert count, ragged token counts and widths
smaller than one tile."""
import numpy as np
import pytest
import torch

from _harness import DEV, GpuRun, WORKLOADS, assert_close, check_routing_equal, f64, oracle_cfg
from mixture_experts_layer_86_b300 import _native as N
from mixture_experts_layer_86_b300 import layer as L
from mixture_experts_layer_86_b300.inputs import Workload, make_inputs
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu


def _full_check(wl, inp=None):
    run = GpuRun(wl, training=True, inp=inp)
    g = run.oracle_route()
    check_routing_equal(run, g)
    inp = run.inp
    lb = None if inp.logit_bias is None else f64(inp.logit_bias)
    ref = O.forward(oracle_cfg(wl), f64(inp.x), f64(inp.w_gate), f64(inp.w1), f64(inp.b1),
                    f64(inp.w2), f64(inp.b2), logit_bias=lb, logits=f64(run.bufs["logits"]))
    assert_close(f64(run.y), ref["y"], wl.dtype, "y")
    assert N.moe_get_device_error() == 0
    return run, ref


def test_empty_batch():
    wl = Workload("empty", 0, 64, 128, 4, 2, 1.0, 4, True, "gelu_tanh", "bf16", seed=0)
    cfg = N.config_from_workload(wl)
    x = torch.empty((1, 64), dtype=torch.bfloat16, device=DEV)
    inp = make_inputs(wl.scaled(1)).to(DEV)
    bufs = L.alloc_buffers(N.config_from_workload(wl.scaled(1)), DEV)
    ws = L.alloc_workspace(N.config_from_workload(wl.scaled(1)), DEV)
    y = torch.empty_like(x)
    bufs["kept_cnt"].fill_(-7)
    N.moe_forward(cfg, x, inp.w_gate, None, inp.w1, inp.b1, inp.w2, inp.b2, y, bufs, ws)
    torch.cuda.synchronize()
    assert bufs["kept_cnt"].tolist() == [0, 0, 0, 0]
    assert bufs["expert_offsets"].tolist() == [0, 0, 0, 0, 0]
    assert float(bufs["l_aux"].item()) == 0.0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_single_token(dtype):
    wl = Workload("one", 1, 64, 128, 2, 2, 1.0, 1, True, "gelu_tanh", dtype, seed=3, bias_std=0.1)
    _full_check(wl)


def test_all_tokens_prefer_one_expert():
    wl = Workload("hot", 1000, 128, 256, 8, 2, 1.0, 4, True, "gelu_tanh", "bf16", seed=5,
                  bias_std=0.1)
    inp = make_inputs(wl)
    inp.logit_bias = torch.tensor([0, 0, 0, 30.0, 0, 0, 0, 0])
    run, ref = _full_check(wl, inp)
    rt = ref["routing"]
    assert rt.routed[3] == 1000 and rt.kept[3] == rt.capacity == 250
    assert (rt.slot[:, 0] < 0).sum() == 750


def test_no_cap_heavy_skew_multi_tile():
    wl = Workload("skew_nocap", 1500, 256, 512, 6, 2, 1.0, 4, False, "gelu_tanh", "bf16",
                  seed=6, skew=3.0, bias_std=0.1)
    run, ref = _full_check(wl)
    assert ref["routing"].kept.max() > 3 * 128      # several m-tiles for one expert
    assert (ref["routing"].slot >= 0).all()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_single_expert_is_dense_ffn(dtype):
    wl = Workload("e1", 333, 64, 192, 1, 1, 1.0, 4, True, "relu", dtype, seed=8, bias_std=0.1)
    run, ref = _full_check(wl)
    inp = run.inp
    dense = O.activation(f64(inp.x) @ f64(inp.w1[0]).T + f64(inp.b1[0]), "relu") \
        @ f64(inp.w2[0]).T + f64(inp.b2[0])
    assert_close(f64(run.y), dense, dtype, "dense")


def test_max_experts():
    wl = Workload("e256", 3000, 64, 128, 256, 2, 1.5, 2, True, "gelu_tanh", "bf16", seed=9,
                  bias_std=0.1)
    _full_check(wl)


@pytest.mark.parametrize("S", [127, 129, 1001])
def test_ragged_batches_k1_bf16(S):
    wl = Workload("ragged", S, 96, 160, 5, 1, 1.1, 3, True, "gelu_erf", "bf16", seed=S,
                  bias_std=0.1)
    _full_check(wl)
