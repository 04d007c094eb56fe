"""Shared helpers of the GPU parity tests: run the CUDA path through the C
ABI, convert its tensors to float64 / int64 exactly, and evaluate the oracle
on the same inputs.  Tolerances are the layer's specification:
  fp32 layer: max|err| <= 1e-5 * max|ref|
  bf16 layer: rel L2 <= 5e-3 and max|err| <= 2e-2 * max|ref|
"""
from __future__ import annotations

import numpy as np
import torch

from mixture_experts_layer_86_b300 import _native as N
from mixture_experts_layer_86_b300 import layer as L
from mixture_experts_layer_86_b300.inputs import WORKLOADS, Workload, make_inputs
from oracle import moe_oracle as O

DEV = "cuda:0"
_INPUT_CACHE = {}


def f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def i64(t):
    return t.detach().to("cpu").numpy().astype(np.int64)


def inputs_for(wl: Workload):
    """CPU inputs of a workload, cached for the session (full-size draws are slow)."""
    key = wl
    if key not in _INPUT_CACHE:
        if len(_INPUT_CACHE) > 4:
            _INPUT_CACHE.clear()
        _INPUT_CACHE[key] = make_inputs(wl)
    return _INPUT_CACHE[key]


def oracle_cfg(wl: Workload) -> O.LayerConfig:
    return O.LayerConfig(wl.num_tokens, wl.hidden_size, wl.ffn_size, wl.num_experts, wl.k,
                         wl.capacity_factor, wl.min_capacity, wl.drop_tokens, wl.act,
                         wl.aux_loss_weight, wl.gate_temperature, wl.aux_loss_type)


class GpuRun:
    """One forward (and optionally backward) of the CUDA path."""

    def __init__(self, wl: Workload, training: bool = False, inp=None):
        self.wl = wl
        self.cfg = N.config_from_workload(wl)
        self.inp = inp if inp is not None else inputs_for(wl)
        self.d = self.inp.to(DEV)
        self.training = training
        self.y, self.l_aux, self.kept, self.bufs = L.forward(
            self.cfg, self.d.x, self.d.w_gate, self.d.logit_bias, self.d.w1, self.d.b1,
            self.d.w2, self.d.b2, training=training)
        torch.cuda.synchronize()
        self.grads = None

    def backward(self):
        self.grads = L.backward(self.cfg, self.d.x, self.d.w_gate, self.d.w1, self.d.w2,
                                self.bufs, self.d.dy)
        torch.cuda.synchronize()
        return self.grads

    @property
    def num_rows(self) -> int:
        return int(self.bufs["expert_offsets"][-1].item())

    def oracle_route(self) -> dict:
        """Oracle routing of the GPU's own fp32 logits (widened exactly)."""
        return O.route(f64(self.bufs["logits"]), oracle_cfg(self.wl))


def check_routing_equal(run: GpuRun, g: dict):
    rt = g["routing"]
    b = run.bufs
    assert np.array_equal(i64(b["topk_idx"]), rt.idx), "topk_idx"
    assert np.array_equal(i64(b["slot"]), rt.slot), "slot"
    assert np.array_equal(i64(b["routed_cnt"]), rt.routed), "routed_cnt"
    assert np.array_equal(i64(b["kept_cnt"]), rt.kept), "kept_cnt"
    assert np.array_equal(i64(b["expert_offsets"]), rt.offsets), "expert_offsets"
    R = rt.num_rows
    assert np.array_equal(i64(b["row_src"])[:R], rt.row_src), "row_src"


def assert_close(got, ref, dtype: str, what: str = ""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    if ref.size == 0:
        return {}
    max_rel = float(err.max()) / scale if scale > 0 else float(err.max())
    rel_l2 = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    if dtype == "f32":
        assert max_rel <= 1e-5, f"{what}: max|err|/max|ref| = {max_rel:.3e}"
    else:
        assert rel_l2 <= 5e-3, f"{what}: rel L2 = {rel_l2:.3e}"
        assert max_rel <= 2e-2, f"{what}: max|err|/max|ref| = {max_rel:.3e}"
    return {"max_rel": max_rel, "rel_l2": rel_l2}


class ErrAcc:
    """assert_close over an array compared piece by piece (for instance one
    expert's rows at a time): the norms and maxima are accumulated, so the
    verdict is the one assert_close gives on the whole array."""

    def __init__(self, what: str):
        self.what = what
        self.se = self.sr = 0.0
        self.max_err = self.max_ref = 0.0
        self.n = 0

    def add(self, got, ref):
        got = np.asarray(got, np.float64)
        ref = np.asarray(ref, np.float64)
        assert got.shape == ref.shape, (self.what, got.shape, ref.shape)
        if ref.size == 0:
            return
        assert np.all(np.isfinite(got)), f"{self.what}: non-finite values"
        d = got - ref
        self.se += float(np.sum(d * d))
        self.sr += float(np.sum(ref * ref))
        self.max_err = max(self.max_err, float(np.abs(d).max()))
        self.max_ref = max(self.max_ref, float(np.abs(ref).max()))
        self.n += ref.size

    def check(self, dtype: str):
        if self.n == 0:
            return {}
        max_rel = self.max_err / self.max_ref if self.max_ref > 0 else self.max_err
        rel_l2 = float(np.sqrt(self.se) / max(np.sqrt(self.sr), 1e-300))
        if dtype == "f32":
            assert max_rel <= 1e-5, f"{self.what}: max|err|/max|ref| = {max_rel:.3e}"
        else:
            assert rel_l2 <= 5e-3, f"{self.what}: rel L2 = {rel_l2:.3e}"
            assert max_rel <= 2e-2, f"{self.what}: max|err|/max|ref| = {max_rel:.3e}"
        return {"max_rel": max_rel, "rel_l2": rel_l2, "n": self.n}


def topk_margin(logits: np.ndarray, k: int) -> np.ndarray:
    """Per token: the smallest gap that decides its choices (k-th vs
    (k+1)-th, and for k=2 also 1st vs 2nd)."""
    srt = -np.sort(-logits, axis=1)
    m = srt[:, k - 1] - srt[:, k] if logits.shape[1] > k else np.full(len(logits), np.inf)
    if k == 2:
        m = np.minimum(m, srt[:, 0] - srt[:, 1])
    return m
