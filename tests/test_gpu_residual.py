"""GPU parity of the PR-MoE layer (moe_forward_residual): y = MoE(x) +
MLP(x) with a dense MLP on every token, or, with the learned mix,
y = c0 MoE(x) + c1 MLP(x), c = softmax(x W_c^T + b_c) per token (reading R8
of the oracle).  Routing must equal the plain layer's; y, the MLP's output
and c are compared with the float64 oracle (fp32 layer: max|err| <= 1e-5
max|ref|; bf16: rel L2 <= 5e-3, max|err| <= 2e-2 max|ref|; c: fp32 dot
products of bf16-exact inputs, max|err| <= 2e-6)."""
import types

import numpy as np
import pytest
import torch

from _harness import DEV, WORKLOADS, assert_close, check_routing_equal, f64, oracle_cfg
from mixture_experts_layer_86_b300 import _native as N
from mixture_experts_layer_86_b300 import layer as L
from mixture_experts_layer_86_b300.inputs import make_inputs, make_residual_mix, make_residual_weights
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu


def _run(wl, mix=None):
    inp = make_inputs(wl)
    res = make_residual_weights(wl)
    d = inp.to(DEV)
    rw = [t.to(DEV) for t in res]
    cfg = N.config_from_workload(wl)
    mw, mb = (None, None) if mix is None else [t.to(DEV) for t in mix]
    y, l_aux, kept, st = L.forward_residual(cfg, d.x, d.w_gate, d.logit_bias, d.w1, d.b1, d.w2,
                                            d.b2, *rw, mix_w=mw, mix_b=mb)
    torch.cuda.synchronize()
    assert N.moe_get_device_error() == 0
    return inp, res, y, st


@pytest.mark.parametrize("name,S", [("tiny_fp32", 256), ("e8_bf16", 1000), ("e64_bf16", 300),
                                    ("skew_e16_nodrop", 500), ("decode_e64", 256)])
def test_residual_forward_parity(name, S):
    wl = WORKLOADS[name].scaled(S, bias_std=0.1)
    inp, res, y, st = _run(wl)
    c = oracle_cfg(wl)
    lb = None if inp.logit_bias is None else f64(inp.logit_bias)
    ref = O.forward_residual(c, f64(inp.x), None, f64(inp.w1), f64(inp.b1), f64(inp.w2),
                             f64(inp.b2), *[f64(t) for t in res], logit_bias=lb,
                             logits=f64(st["logits"]))
    # the routing is the plain layer's
    g = O.route(f64(st["logits"]), c)
    check_routing_equal(types.SimpleNamespace(bufs=st), g)
    assert_close(f64(st["res_out"]), ref["residual"], wl.dtype, "residual MLP")
    assert_close(f64(y), ref["y"], wl.dtype, "y")


def test_residual_forward_full_size_sampled():
    wl = WORKLOADS["e64_bf16"]
    inp, res, y, st = _run(wl)
    c = oracle_cfg(wl)
    g = O.route(f64(st["logits"]), c)
    rt = g["routing"]
    gen = np.random.default_rng(3)
    toks = sorted(set([0, wl.num_tokens - 1]) | set(gen.choice(wl.num_tokens, 24, replace=False).tolist()))
    x = f64(inp.x)[toks]
    want = O.residual_mlp(x, *[f64(t) for t in res], wl.act)
    for i, s in enumerate(toks):
        for j in range(wl.k):
            if rt.slot[s, j] < 0:
                continue
            e = int(rt.idx[s, j])
            _, _, o = O.expert_ffn(x[i:i + 1], np.array([0, 1]), f64(inp.w1[e:e + 1]),
                                   f64(inp.b1[e:e + 1]), f64(inp.w2[e:e + 1]), f64(inp.b2[e:e + 1]),
                                   wl.act)
            want[i] += g["weights"][s, j] * o[0]
    assert_close(f64(y[toks]), want, wl.dtype, "y sampled")


@pytest.mark.parametrize("name,S", [("tiny_fp32", 256), ("e8_bf16", 1000), ("e64_bf16", 300),
                                    ("skew_e16_nodrop", 500), ("decode_e64", 256)])
def test_residual_learned_mix_parity(name, S):
    wl = WORKLOADS[name].scaled(S, bias_std=0.1)
    mix = make_residual_mix(wl)
    inp, res, y, st = _run(wl, mix)
    c = oracle_cfg(wl)
    lb = None if inp.logit_bias is None else f64(inp.logit_bias)
    ref = O.forward_residual(c, f64(inp.x), None, f64(inp.w1), f64(inp.b1), f64(inp.w2),
                             f64(inp.b2), *[f64(t) for t in res], logit_bias=lb,
                             logits=f64(st["logits"]), coef_w=f64(mix[0]), coef_b=f64(mix[1]))
    g = O.route(f64(st["logits"]), c)
    check_routing_equal(types.SimpleNamespace(bufs=st), g)
    assert np.abs(f64(st["mix"]) - ref["coef"]).max() <= 2e-6
    # both branches really take part: c is neither 0 nor 1 anywhere near all tokens
    assert 0.05 < float(ref["coef"][:, 0].mean()) < 0.95
    assert_close(f64(st["res_out"]), ref["residual"], wl.dtype, "residual MLP")
    assert_close(f64(y), ref["y"], wl.dtype, "y")


def test_residual_learned_mix_full_size_sampled():
    wl = WORKLOADS["e64_bf16"]
    mix = make_residual_mix(wl)
    inp, res, y, st = _run(wl, mix)
    c = oracle_cfg(wl)
    g = O.route(f64(st["logits"]), c)
    rt = g["routing"]
    gen = np.random.default_rng(4)
    toks = sorted(set([0, wl.num_tokens - 1]) | set(gen.choice(wl.num_tokens, 24, replace=False).tolist()))
    x = f64(inp.x)[toks]
    cf = O.residual_coef(x, f64(mix[0]), f64(mix[1]))
    assert np.abs(f64(st["mix"])[toks] - cf).max() <= 2e-6
    want = cf[:, 1:2] * O.residual_mlp(x, *[f64(t) for t in res], wl.act)
    for i, s in enumerate(toks):
        for j in range(wl.k):
            if rt.slot[s, j] < 0:
                continue
            e = int(rt.idx[s, j])
            _, _, o = O.expert_ffn(x[i:i + 1], np.array([0, 1]), f64(inp.w1[e:e + 1]),
                                   f64(inp.b1[e:e + 1]), f64(inp.w2[e:e + 1]), f64(inp.b2[e:e + 1]),
                                   wl.act)
            want[i] += cf[i, 0] * g["weights"][s, j] * o[0]
    assert_close(f64(y[toks]), want, wl.dtype, "y sampled")
