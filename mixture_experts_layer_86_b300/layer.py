"""Allocation helpers around the C ABI: the caller-side memory plan of one
MoE layer call (torch allocates, the library computes).

``forward`` returns ``(y, l_aux, expert_count, state)`` like MoE.forward's
``(output, gate_loss, expert_count)`` on the deepspeed.moe overview page
(§2.1); ``backward`` returns the gradients of <dY, y> + aux_loss_weight*l_aux.
"""
from __future__ import annotations

import torch

from . import _native as N


def torch_dtype(cfg: N.MoeConfig) -> torch.dtype:
    return torch.float32 if cfg.dtype == N.MOE_F32 else torch.bfloat16


def alloc_buffers(cfg: N.MoeConfig, device, training: bool = False,
                  fused_dispatch: bool = False) -> dict:
    """Device buffers of one forward pass, sized from the config alone.  With
    fused_dispatch (bf16 inference) there is no x_disp: moe_forward then reads
    the experts' token rows straight from x inside the first expert GEMM."""
    S, E, k = cfg.num_tokens, cfg.num_experts, cfg.k
    d, f = cfg.hidden_size, cfg.ffn_size
    R = N.moe_max_rows(cfg)
    dt = torch_dtype(cfg)
    i32 = dict(dtype=torch.int32, device=device)
    f32 = dict(dtype=torch.float32, device=device)
    return {
        "logits": torch.empty((S, E), **f32),
        "probs": torch.empty((S, E), **f32) if training else None,
        "topk_idx": torch.empty((S, k), **i32),
        "topk_w": torch.empty((S, k), **f32),
        "slot": torch.empty((S, k), **i32),
        "routed_cnt": torch.empty((E,), **i32),
        "kept_cnt": torch.empty((E,), **i32),
        "expert_offsets": torch.empty((E + 1,), **i32),
        "row_src": torch.empty((max(R, 1),), **i32),
        "l_aux": torch.empty((1,), **f32),
        "x_disp": None if fused_dispatch else torch.empty((max(R, 1), d), dtype=dt, device=device),
        "h_pre": torch.empty((max(R, 1), f), dtype=dt, device=device) if training else None,
        "h": torch.empty((max(R, 1), f), dtype=dt, device=device),
        "out_disp": torch.empty((max(R, 1), d), dtype=dt, device=device),
    }


def alloc_workspace(cfg: N.MoeConfig, device, for_backward: bool = False) -> torch.Tensor:
    n = N.moe_workspace_size(cfg, for_backward)
    return torch.empty((max(n, 256),), dtype=torch.uint8, device=device)


def forward(cfg, x, w_gate, logit_bias, w1, b1, w2, b2, bufs=None, workspace=None,
            y=None, training=False, stream=None, fused_dispatch=False):
    dev = x.device
    if bufs is None:
        bufs = alloc_buffers(cfg, dev, training, fused_dispatch=fused_dispatch and not training)
    if workspace is None:
        workspace = alloc_workspace(cfg, dev)
    if y is None:
        y = torch.empty_like(x)
    N.moe_forward(cfg, x, w_gate, logit_bias, w1, b1, w2, b2, y, bufs, workspace, stream)
    return y, bufs["l_aux"], bufs["kept_cnt"], bufs


def forward_residual(cfg, x, w_gate, logit_bias, w1, b1, w2, b2, rw1, rb1, rw2, rb2,
                     bufs=None, workspace=None, y=None, stream=None, mix_w=None, mix_b=None):
    """PR-MoE layer (``use_residual=True``): y = MoE(x) + MLP(x) with the
    dense MLP weights rw1 [f,d], rb1 [f], rw2 [d,f], rb2 [d]; with the mixing
    weights mix_w [2,d], mix_b [2] given, y = c0 MoE(x) + c1 MLP(x) with
    c = softmax(x mix_w^T + mix_b) per token.  Returns (y, l_aux,
    expert_count, state); state also holds the MLP's activation ("res_h"),
    output ("res_out") and, with the mix, c ("mix", [S,2] fp32)."""
    dev = x.device
    if bufs is None:
        bufs = alloc_buffers(cfg, dev)
    if workspace is None:
        workspace = alloc_workspace(cfg, dev)
    if y is None:
        y = torch.empty_like(x)
    dt = torch_dtype(cfg)
    res_h = torch.empty((cfg.num_tokens, cfg.ffn_size), dtype=dt, device=dev)
    res_out = torch.empty((cfg.num_tokens, cfg.hidden_size), dtype=dt, device=dev)
    mix = None
    if mix_w is not None:
        mix = torch.empty((cfg.num_tokens, 2), dtype=torch.float32, device=dev)
    N.moe_forward_residual(cfg, x, w_gate, logit_bias, w1, b1, w2, b2, rw1, rb1, rw2, rb2, y,
                           bufs, res_h, res_out, workspace, stream, mix_w=mix_w, mix_b=mix_b,
                           mix=mix)
    state = dict(bufs, res_h=res_h, res_out=res_out, mix=mix)
    return y, bufs["l_aux"], bufs["kept_cnt"], state


def backward(cfg, x, w_gate, w1, w2, bufs, dy, workspace=None, grads=None, stream=None):
    dev = x.device
    if workspace is None:
        workspace = alloc_workspace(cfg, dev, for_backward=True)
    if grads is None:
        grads = {"dx": torch.empty_like(x), "dw_gate": torch.empty_like(w_gate),
                 "dw1": torch.empty_like(w1), "db1": torch.empty(w1.shape[:2], dtype=w1.dtype, device=dev),
                 "dw2": torch.empty_like(w2), "db2": torch.empty(w2.shape[:2], dtype=w2.dtype, device=dev)}
    N.moe_backward(cfg, x, w_gate, w1, w2, bufs, dy, grads["dx"], grads["dw_gate"], grads["dw1"],
                   grads["db1"], grads["dw2"], grads["db2"], workspace, stream)
    return grads


class HostPipeline:
    """Forward passes over batches that live in (pinned) host memory, with the
    host-to-device copy of the next batch and the device-to-host copy of the
    previous result running on their own streams while the current forward
    runs: two buffer slots, three streams, ordered by CUDA events.  This is
    stream and buffer bookkeeping only; every step of the layer runs in the
    library's kernels (``moe_forward``).

    ``submit(x_host, y_host, laux_host=None, count_host=None)`` enqueues one
    batch and returns at once; ``synchronize()`` waits for every result.  A
    host output buffer may be reused once the submit that wrote it is two or
    more calls back and its copy has finished (``synchronize``, or the
    event returned by ``submit``)."""

    def __init__(self, cfg, w_gate, logit_bias, w1, b1, w2, b2, device):
        self.cfg = cfg
        self.weights = (w_gate, logit_bias, w1, b1, w2, b2)
        dt = torch_dtype(cfg)
        shape = (cfg.num_tokens, cfg.hidden_size)
        self.slots = [{"x": torch.empty(shape, dtype=dt, device=device),
                       "y": torch.empty(shape, dtype=dt, device=device),
                       "bufs": alloc_buffers(cfg, device),
                       "ev_in": torch.cuda.Event(), "ev_comp": torch.cuda.Event(),
                       "ev_out": torch.cuda.Event(), "used": False} for _ in range(2)]
        for sl in self.slots:
            sl["bufs"]["logits"] = None    # the gate's optional output; never copied out
        self.workspace = alloc_workspace(cfg, device)
        self.s_in = torch.cuda.Stream(device)
        self.s_comp = torch.cuda.Stream(device)
        self.s_out = torch.cuda.Stream(device)
        self.n = 0

    def submit(self, x_host, y_host, laux_host=None, count_host=None):
        sl = self.slots[self.n % 2]
        if sl["used"]:
            self.s_in.wait_event(sl["ev_comp"])      # the slot's last forward has read x
        with torch.cuda.stream(self.s_in):
            sl["x"].copy_(x_host, non_blocking=True)
            sl["ev_in"].record(self.s_in)
        self.s_comp.wait_event(sl["ev_in"])
        if sl["used"]:
            self.s_comp.wait_event(sl["ev_out"])     # the slot's last result is copied out
        w_gate, logit_bias, w1, b1, w2, b2 = self.weights
        N.moe_forward(self.cfg, sl["x"], w_gate, logit_bias, w1, b1, w2, b2, sl["y"],
                      sl["bufs"], self.workspace, self.s_comp)
        sl["ev_comp"].record(self.s_comp)
        self.s_out.wait_event(sl["ev_comp"])
        with torch.cuda.stream(self.s_out):
            y_host.copy_(sl["y"], non_blocking=True)
            if laux_host is not None:
                laux_host.copy_(sl["bufs"]["l_aux"], non_blocking=True)
            if count_host is not None:
                count_host.copy_(sl["bufs"]["kept_cnt"], non_blocking=True)
            sl["ev_out"].record(self.s_out)
        sl["used"] = True
        self.n += 1
        return sl["ev_out"]

    def synchronize(self):
        for s in (self.s_in, self.s_comp, self.s_out):
            s.synchronize()
