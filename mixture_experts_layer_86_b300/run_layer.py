"""Runs the MoE layer a few times on cuda:0 through the C ABI -- a fixed,
small command for profilers and quick checks.

    python -m mixture_experts_layer_86_b300.run_layer --workload e64_bf16 \\
        [--tokens S] [--experts E] [--iters N] [--backward]

--tokens / --experts shrink the batch / the number of experts of a named
workload while keeping the per-expert shape (d, f, k, capacity factor).
"""
from __future__ import annotations

import argparse
import dataclasses

import torch

from . import _native as N
from . import layer as L
from .inputs import WORKLOADS, make_inputs


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="e64_bf16")
    ap.add_argument("--tokens", type=int, default=None)
    ap.add_argument("--experts", type=int, default=None)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--backward", action="store_true")
    a = ap.parse_args()
    wl = WORKLOADS[a.workload]
    if a.experts is not None:
        wl = dataclasses.replace(wl, num_experts=a.experts)
    if a.tokens is not None:
        wl = wl.scaled(a.tokens)
    inp = make_inputs(wl, with_dy=a.backward).to("cuda:0")
    cfg = N.config_from_workload(wl)
    bufs = L.alloc_buffers(cfg, "cuda:0", training=a.backward)
    ws = L.alloc_workspace(cfg, "cuda:0", for_backward=False)
    wsb = L.alloc_workspace(cfg, "cuda:0", for_backward=True) if a.backward else None
    for _ in range(a.iters):
        y, l_aux, kept, _ = L.forward(cfg, inp.x, inp.w_gate, inp.logit_bias, inp.w1, inp.b1,
                                      inp.w2, inp.b2, bufs=bufs, workspace=ws)
        if a.backward:
            L.backward(cfg, inp.x, inp.w_gate, inp.w1, inp.w2, bufs, inp.dy, workspace=wsb)
    torch.cuda.synchronize()
    err = N.moe_get_device_error()
    print(f"{wl.name}: rows={int(bufs['expert_offsets'][-1])} l_aux={float(l_aux):.5f} "
          f"device_error={err:#x}")
    if err:
        raise SystemExit(1)


if __name__ == "__main__":
    main()
