"""GPU check of HostPipeline, the host-batch stream pipeline: with the
host-to-device copy, the forward and the device-to-host copy of successive
batches overlapping on three streams and two buffer slots, every batch's
y, l_aux and per-expert counts must be bit-identical to a plain synchronous
moe_forward of that batch (a missing event wait would let a copy read a slot
that another batch is still writing)."""
import dataclasses

import pytest
import torch

from _harness import DEV, WORKLOADS
from mixture_experts_layer_86_b300 import _native as N
from mixture_experts_layer_86_b300 import layer as L
from mixture_experts_layer_86_b300.inputs import make_gate_inputs, make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,S,nb", [("e8_bf16", 1024, 5), ("tiny_fp32", 300, 4),
                                       ("e64_bf16", 4096, 6)])
def test_host_pipeline_matches_sync_forward(name, S, nb):
    wl = WORKLOADS[name].scaled(S)
    cfg = N.config_from_workload(wl)
    d = make_inputs(wl).to(DEV)
    xs = [make_gate_inputs(dataclasses.replace(wl, seed=wl.seed + 17 * (i + 1)))[0].pin_memory()
          for i in range(nb)]
    ys = [torch.empty_like(x).pin_memory() for x in xs]
    la = [torch.empty(1, dtype=torch.float32).pin_memory() for _ in xs]
    cnt = [torch.empty(wl.num_experts, dtype=torch.int32).pin_memory() for _ in xs]

    pipe = L.HostPipeline(cfg, d.w_gate, d.logit_bias, d.w1, d.b1, d.w2, d.b2, DEV)
    for i in range(nb):
        pipe.submit(xs[i], ys[i], la[i], cnt[i])
    pipe.synchronize()

    for i in range(nb):
        y, l_aux, kept, _ = L.forward(cfg, xs[i].to(DEV), d.w_gate, d.logit_bias, d.w1, d.b1,
                                      d.w2, d.b2)
        torch.cuda.synchronize()
        assert torch.equal(ys[i], y.cpu()), f"batch {i}: y differs"
        assert torch.equal(la[i], l_aux.cpu()), f"batch {i}: l_aux differs"
        assert torch.equal(cnt[i], kept.cpu()), f"batch {i}: counts differ"
    assert N.moe_get_device_error() == 0
