"""The give-up path of a bounded device wait, on the GPU, without a fault: a
1 ns limit on the single-launch gate's progress waits makes them run out;
the kernel records its code in the device error word, drains its own copies
and MMAs and returns (outputs unspecified but in range); with the default
limit restored the next call computes exactly what it did before."""
import pytest
import torch

from mixture_experts_layer_86_b300 import _native as N
from mixture_experts_layer_86_b300 import layer as L
from mixture_experts_layer_86_b300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GATE_CODES = {0x05, 0x06, 0x07, 0x0C}   # producer, MMA, epilogue, grid barrier of the gate


def _gate(cfg, inp, bufs, ws):
    N.moe_gate_topk(cfg, inp.x, inp.w_gate, inp.logit_bias, bufs["logits"], bufs["probs"],
                    bufs["topk_idx"], bufs["topk_w"], bufs["slot"], bufs["routed_cnt"],
                    bufs["kept_cnt"], bufs["expert_offsets"], bufs["row_src"], bufs["l_aux"], ws)
    torch.cuda.synchronize()


def test_gate_wait_gives_up_records_its_code_and_recovers():
    wl = WORKLOADS["e64_bf16"].scaled(8192)
    cfg = N.config_from_workload(wl)
    inp = make_inputs(wl).to(DEV)
    ws = L.alloc_workspace(cfg, DEV)
    ref = L.alloc_buffers(cfg, DEV, training=True)
    _gate(cfg, inp, ref, ws)
    assert N.moe_get_device_error() == 0
    got = L.alloc_buffers(cfg, DEV, training=True)
    try:
        N.moe_debug_set_wait_limit(1)
        _gate(cfg, inp, got, ws)
        code = N.moe_get_device_error()
    finally:
        N.moe_debug_set_wait_limit(0)
    assert code != 0 and (code >> 24) in GATE_CODES, hex(code)
    # whatever the kernel left is in range
    E, cap, S = wl.num_experts, N.moe_capacity(cfg), wl.num_tokens
    idx, slot, off = got["topk_idx"], got["slot"], got["expert_offsets"]
    assert int(idx.min()) >= 0 and int(idx.max()) < E
    assert int(slot.min()) >= -1 and int(slot.max()) < cap
    assert bool((off[1:] >= off[:-1]).all()) and 0 <= int(off[-1]) <= N.moe_max_rows(cfg)
    # the context is fine and the next call with the default limit is exact
    again = L.alloc_buffers(cfg, DEV, training=True)
    _gate(cfg, inp, again, ws)
    assert N.moe_get_device_error() == 0
    for key in ("logits", "probs", "topk_idx", "topk_w", "slot", "routed_cnt", "kept_cnt",
                "expert_offsets", "l_aux"):
        assert torch.equal(again[key], ref[key]), key
    R = int(ref["expert_offsets"][-1])
    assert torch.equal(again["row_src"][:R], ref["row_src"][:R])
    assert S == idx.shape[0]
