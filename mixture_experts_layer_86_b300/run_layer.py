"""Runs the MoE layer (or one of its stages) a few times on cuda:0 through
the C ABI -- a fixed, small command for profilers and quick checks.

    python -m mixture_experts_layer_86_b300.run_layer --workload e64_bf16 \\
        [--tokens S] [--experts E] [--iters N] [--backward] [--fused] [--stage gate]

--tokens / --experts shrink the batch / the number of experts of a named
workload while keeping the per-expert shape (d, f, k, capacity factor).
--fused runs the forward without the x_disp copy (the dispatch fused into the
first expert GEMM; bf16 forward only).
--stage gate runs only moe_gate_topk and allocates only what it needs (x,
W_g, the routing outputs and the workspace), so a profiler that saves and
restores device memory between its passes has little to move.
"""
from __future__ import annotations

import argparse
import dataclasses

import torch

from . import _native as N
from . import layer as L
from .inputs import WORKLOADS, make_gate_inputs, make_inputs


def run_gate(wl, iters):
    cfg = N.config_from_workload(wl)
    S, E, k = wl.num_tokens, wl.num_experts, wl.k
    x, w_gate, bias = make_gate_inputs(wl)
    x, w_gate = x.cuda(), w_gate.cuda()
    bias = None if bias is None else bias.cuda()
    i32 = dict(dtype=torch.int32, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    R = max(N.moe_max_rows(cfg), 1)
    out = dict(logits=torch.empty((S, E), **f32), idx=torch.empty((S, k), **i32),
               w=torch.empty((S, k), **f32), slot=torch.empty((S, k), **i32),
               routed=torch.empty(E, **i32), kept=torch.empty(E, **i32),
               offsets=torch.empty(E + 1, **i32), rows=torch.empty(R, **i32),
               l_aux=torch.empty(1, **f32))
    ws = L.alloc_workspace(cfg, "cuda")
    for _ in range(iters):
        N.moe_gate_topk(cfg, x, w_gate, bias, out["logits"], None, out["idx"], out["w"],
                        out["slot"], out["routed"], out["kept"], out["offsets"], out["rows"],
                        out["l_aux"], ws)
    torch.cuda.synchronize()
    return int(out["offsets"][-1]), float(out["l_aux"])


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="e64_bf16")
    ap.add_argument("--tokens", type=int, default=None)
    ap.add_argument("--experts", type=int, default=None)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--backward", action="store_true")
    ap.add_argument("--fused", action="store_true")
    ap.add_argument("--stage", default="forward", choices=["forward", "gate"])
    a = ap.parse_args()
    wl = WORKLOADS[a.workload]
    if a.experts is not None:
        wl = dataclasses.replace(wl, num_experts=a.experts)
    if a.tokens is not None:
        wl = wl.scaled(a.tokens)
    if a.stage == "gate":
        rows, l_aux = run_gate(wl, a.iters)
    else:
        inp = make_inputs(wl, with_dy=a.backward).to("cuda:0")
        cfg = N.config_from_workload(wl)
        bufs = L.alloc_buffers(cfg, "cuda:0", training=a.backward,
                               fused_dispatch=a.fused and not a.backward)
        ws = L.alloc_workspace(cfg, "cuda:0", for_backward=False)
        wsb = L.alloc_workspace(cfg, "cuda:0", for_backward=True) if a.backward else None
        for _ in range(a.iters):
            y, l_aux_t, kept, _ = L.forward(cfg, inp.x, inp.w_gate, inp.logit_bias, inp.w1,
                                            inp.b1, inp.w2, inp.b2, bufs=bufs, workspace=ws)
            if a.backward:
                L.backward(cfg, inp.x, inp.w_gate, inp.w1, inp.w2, bufs, inp.dy, workspace=wsb)
        torch.cuda.synchronize()
        rows, l_aux = int(bufs["expert_offsets"][-1]), float(l_aux_t)
    err = N.moe_get_device_error()
    print(f"{wl.name} [{a.stage}]: rows={rows} l_aux={l_aux:.5f} device_error={err:#x}")
    if err:
        raise SystemExit(1)


if __name__ == "__main__":
    main()
