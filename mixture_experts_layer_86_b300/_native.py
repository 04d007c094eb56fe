"""ctypes binding of ``libmoe_b300.so`` (declared in ``include/moe_b300.h``).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  Functions carry the C names; tensors are passed as device
pointers (``Tensor.data_ptr()``), ``None`` becomes NULL, and the stream
defaults to torch's current stream.  A non-OK status raises ``MoeError``.
If the library has not been built, importing this module raises -- there is
no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_double, c_float, c_int, c_int32, c_int64, c_size_t, c_uint32, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_b300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_DEVICE = range(6)
MOE_F32, MOE_BF16 = 0, 1
MOE_ACT_RELU, MOE_ACT_GELU_TANH, MOE_ACT_GELU_ERF = 0, 1, 2
MOE_AUX_LOAD, MOE_AUX_STD = 0, 1
AUX_CODES = {"load": MOE_AUX_LOAD, "std": MOE_AUX_STD}
MOE_NOISE_NONE, MOE_NOISE_JITTER, MOE_NOISE_RSAMPLE = 0, 1, 2
NOISE_CODES = {"none": MOE_NOISE_NONE, "jitter": MOE_NOISE_JITTER, "rsample": MOE_NOISE_RSAMPLE}
ACT_CODES = {"relu": MOE_ACT_RELU, "gelu_tanh": MOE_ACT_GELU_TANH, "gelu_erf": MOE_ACT_GELU_ERF}
DTYPE_CODES = {"f32": MOE_F32, "bf16": MOE_BF16}


class MoeConfig(ctypes.Structure):
    _fields_ = [("num_tokens", c_int64), ("hidden_size", c_int32), ("ffn_size", c_int32),
                ("num_experts", c_int32), ("k", c_int32), ("capacity_factor", c_double),
                ("min_capacity", c_int32), ("drop_tokens", c_int32), ("act", c_int32),
                ("dtype", c_int32), ("aux_loss_weight", c_float), ("gate_temperature", c_float),
                ("aux_loss_type", c_int32), ("logit_bias_per_token", c_int32),
                ("noise_policy", c_int32), ("second_expert_sampling", c_int32),
                ("use_rts", c_int32), ("jitter_eps", c_float), ("noise_seed", ctypes.c_uint64),
                ("noise_offset", ctypes.c_uint64)]


class MoeBuffers(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in (
        "logits", "probs", "topk_idx", "topk_w", "slot", "routed_cnt", "kept_cnt",
        "expert_offsets", "row_src", "l_aux", "x_disp", "h_pre", "h", "out_disp")]


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {status_string(status)}")
        self.status = status


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      f"`python -m mixture_experts_layer_86_b300.build`")
_lib = ctypes.CDLL(LIB_PATH)

_P = c_void_p
_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [c_int]),
    "moe_capacity": (c_int, [POINTER(MoeConfig), POINTER(c_int64)]),
    "moe_max_rows": (c_int, [POINTER(MoeConfig), POINTER(c_int64)]),
    "moe_workspace_size": (c_int, [POINTER(MoeConfig), c_int, POINTER(c_size_t)]),
    "moe_gate_topk": (c_int, [POINTER(MoeConfig)] + [_P] * 14 + [c_size_t, _P]),
    "moe_route_from_logits": (c_int, [POINTER(MoeConfig)] + [_P] * 11 + [c_size_t, _P]),
    "moe_gate_noise": (c_int, [POINTER(MoeConfig)] + [_P] * 3 + [_P]),
    "moe_gate_topk_static": (c_int, [POINTER(MoeConfig)] + [_P] * 13 + [_P]),
    "moe_dispatch": (c_int, [POINTER(MoeConfig)] + [_P] * 5 + [_P]),
    "moe_expert_ffn": (c_int, [POINTER(MoeConfig)] + [_P] * 9 + [_P]),
    "moe_expert_ffn_gather": (c_int, [POINTER(MoeConfig)] + [_P] * 10 + [_P]),
    "moe_combine": (c_int, [POINTER(MoeConfig)] + [_P] * 6 + [_P]),
    "moe_forward": (c_int, [POINTER(MoeConfig)] + [_P] * 8 + [POINTER(MoeBuffers), _P,
                                                             c_size_t, _P]),
    "moe_forward_residual": (c_int, [POINTER(MoeConfig)] + [_P] * 15 + [POINTER(MoeBuffers)]
                             + [_P] * 3 + [c_size_t, _P]),
    "moe_backward": (c_int, [POINTER(MoeConfig)] + [_P] * 4 + [POINTER(MoeBuffers)] + [_P] * 8
                     + [c_size_t, _P]),
    "moe_get_device_error": (c_int, [POINTER(c_uint32)]),
    "moe_debug_set_wait_limit": (c_int, [ctypes.c_uint64]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def exported_symbols():
    """Names of the C entry points this binding resolved."""
    return sorted(_SIGS)


def library():
    return _lib


def status_string(st: int) -> str:
    return _lib.moe_status_string(int(st)).decode()


def _check(fn: str, st: int):
    if st != MOE_OK:
        raise MoeError(fn, st)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_config(num_tokens, hidden_size, ffn_size, num_experts, k, capacity_factor,
                min_capacity, drop_tokens, act="gelu_tanh", dtype="bf16",
                aux_loss_weight=0.0, gate_temperature=1.0, aux_loss_type="load",
                logit_bias_per_token=False, noise_policy="none",
                second_expert_sampling=False, use_rts=False, jitter_eps=0.01,
                noise_seed=0, noise_offset=0) -> MoeConfig:
    return MoeConfig(int(num_tokens), int(hidden_size), int(ffn_size), int(num_experts), int(k),
                     float(capacity_factor), int(min_capacity), int(bool(drop_tokens)),
                     ACT_CODES[act] if isinstance(act, str) else int(act),
                     DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype),
                     float(aux_loss_weight), float(gate_temperature),
                     AUX_CODES[aux_loss_type] if isinstance(aux_loss_type, str)
                     else int(aux_loss_type), int(bool(logit_bias_per_token)),
                     NOISE_CODES[noise_policy] if isinstance(noise_policy, str)
                     else int(noise_policy), int(bool(second_expert_sampling)),
                     int(bool(use_rts)), float(jitter_eps), int(noise_seed) & (2 ** 64 - 1),
                     int(noise_offset) & (2 ** 64 - 1))


def config_from_workload(wl, num_tokens=None) -> MoeConfig:
    return make_config(wl.num_tokens if num_tokens is None else num_tokens, wl.hidden_size,
                       wl.ffn_size, wl.num_experts, wl.k, wl.capacity_factor, wl.min_capacity,
                       wl.drop_tokens, wl.act, wl.dtype, wl.aux_loss_weight,
                       getattr(wl, "gate_temperature", 1.0), getattr(wl, "aux_loss_type", "load"),
                       getattr(wl, "logit_noise_std", 0.0) > 0,
                       getattr(wl, "noise_policy", "none"),
                       getattr(wl, "second_expert_sampling", False),
                       getattr(wl, "use_rts", False), getattr(wl, "jitter_eps", 0.01),
                       getattr(wl, "noise_seed", 0), getattr(wl, "noise_offset", 0))


# ---------------------------------------------------------------- host-only
def moe_capacity(cfg: MoeConfig) -> int:
    v = c_int64()
    _check("moe_capacity", _lib.moe_capacity(ctypes.byref(cfg), ctypes.byref(v)))
    return v.value


def moe_max_rows(cfg: MoeConfig) -> int:
    v = c_int64()
    _check("moe_max_rows", _lib.moe_max_rows(ctypes.byref(cfg), ctypes.byref(v)))
    return v.value


def moe_workspace_size(cfg: MoeConfig, for_backward: bool = False) -> int:
    v = c_size_t()
    _check("moe_workspace_size",
           _lib.moe_workspace_size(ctypes.byref(cfg), int(bool(for_backward)), ctypes.byref(v)))
    return v.value


# ---------------------------------------------------------------- device calls
def moe_gate_topk(cfg, x, w_gate, logit_bias, logits, probs, topk_idx, topk_w, slot,
                  routed_cnt, kept_cnt, expert_offsets, row_src, l_aux, workspace, stream=None):
    _check("moe_gate_topk", _lib.moe_gate_topk(
        ctypes.byref(cfg), _ptr(x), _ptr(w_gate), _ptr(logit_bias), _ptr(logits), _ptr(probs),
        _ptr(topk_idx), _ptr(topk_w), _ptr(slot), _ptr(routed_cnt), _ptr(kept_cnt),
        _ptr(expert_offsets), _ptr(row_src), _ptr(l_aux), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_gate_topk_static(cfg, x, w_gate, logit_bias, logits, probs, topk_idx, topk_w, slot,
                         routed_cnt, kept_cnt, expert_offsets, row_src, l_aux, stream=None):
    """moe_gate_topk with no workspace argument (scratch compiled into the
    library), for callers that cannot allocate device memory."""
    _check("moe_gate_topk_static", _lib.moe_gate_topk_static(
        ctypes.byref(cfg), _ptr(x), _ptr(w_gate), _ptr(logit_bias), _ptr(logits), _ptr(probs),
        _ptr(topk_idx), _ptr(topk_w), _ptr(slot), _ptr(routed_cnt), _ptr(kept_cnt),
        _ptr(expert_offsets), _ptr(row_src), _ptr(l_aux), _stream(stream)))


def moe_gate_noise(cfg, uniform=None, gumbel=None, position=None, stream=None):
    """The gate's random draws for cfg: uniforms and Gumbel noise [S,E] fp32,
    random-token-selection queue positions [S] int32 (each optional)."""
    _check("moe_gate_noise", _lib.moe_gate_noise(
        ctypes.byref(cfg), _ptr(uniform), _ptr(gumbel), _ptr(position), _stream(stream)))


def moe_route_from_logits(cfg, logits, probs, topk_idx, topk_w, slot, routed_cnt, kept_cnt,
                          expert_offsets, row_src, l_aux, workspace, stream=None):
    _check("moe_route_from_logits", _lib.moe_route_from_logits(
        ctypes.byref(cfg), _ptr(logits), _ptr(probs), _ptr(topk_idx), _ptr(topk_w), _ptr(slot),
        _ptr(routed_cnt), _ptr(kept_cnt), _ptr(expert_offsets), _ptr(row_src), _ptr(l_aux),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_dispatch(cfg, x, topk_idx, slot, expert_offsets, x_disp, stream=None):
    _check("moe_dispatch", _lib.moe_dispatch(
        ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(slot), _ptr(expert_offsets),
        _ptr(x_disp), _stream(stream)))


def moe_expert_ffn(cfg, x_disp, expert_offsets, w1, b1, w2, b2, h_pre, h, out_disp,
                   stream=None):
    _check("moe_expert_ffn", _lib.moe_expert_ffn(
        ctypes.byref(cfg), _ptr(x_disp), _ptr(expert_offsets), _ptr(w1), _ptr(b1), _ptr(w2),
        _ptr(b2), _ptr(h_pre), _ptr(h), _ptr(out_disp), _stream(stream)))


def moe_expert_ffn_gather(cfg, x, row_src, expert_offsets, w1, b1, w2, b2, h_pre, h, out_disp,
                          stream=None):
    """The expert FFN with the dispatch fused into its first GEMM (token rows
    read from x through row_src; no x_disp copy)."""
    _check("moe_expert_ffn_gather", _lib.moe_expert_ffn_gather(
        ctypes.byref(cfg), _ptr(x), _ptr(row_src), _ptr(expert_offsets), _ptr(w1), _ptr(b1),
        _ptr(w2), _ptr(b2), _ptr(h_pre), _ptr(h), _ptr(out_disp), _stream(stream)))


def moe_combine(cfg, out_disp, topk_idx, slot, expert_offsets, topk_w, y, stream=None):
    _check("moe_combine", _lib.moe_combine(
        ctypes.byref(cfg), _ptr(out_disp), _ptr(topk_idx), _ptr(slot), _ptr(expert_offsets),
        _ptr(topk_w), _ptr(y), _stream(stream)))


def buffers_struct(bufs: dict) -> MoeBuffers:
    return MoeBuffers(*[_ptr(bufs.get(n)) for n, _ in MoeBuffers._fields_])


def moe_forward(cfg, x, w_gate, logit_bias, w1, b1, w2, b2, y, bufs, workspace, stream=None):
    b = bufs if isinstance(bufs, MoeBuffers) else buffers_struct(bufs)
    _check("moe_forward", _lib.moe_forward(
        ctypes.byref(cfg), _ptr(x), _ptr(w_gate), _ptr(logit_bias), _ptr(w1), _ptr(b1),
        _ptr(w2), _ptr(b2), _ptr(y), ctypes.byref(b), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_forward_residual(cfg, x, w_gate, logit_bias, w1, b1, w2, b2, rw1, rb1, rw2, rb2, y,
                         bufs, res_h, res_out, workspace, stream=None, mix_w=None, mix_b=None,
                         mix=None):
    b = bufs if isinstance(bufs, MoeBuffers) else buffers_struct(bufs)
    _check("moe_forward_residual", _lib.moe_forward_residual(
        ctypes.byref(cfg), _ptr(x), _ptr(w_gate), _ptr(logit_bias), _ptr(w1), _ptr(b1),
        _ptr(w2), _ptr(b2), _ptr(rw1), _ptr(rb1), _ptr(rw2), _ptr(rb2), _ptr(mix_w), _ptr(mix_b),
        _ptr(mix), _ptr(y), ctypes.byref(b), _ptr(res_h), _ptr(res_out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_backward(cfg, x, w_gate, w1, w2, saved, dy, dx, dw_gate, dw1, db1, dw2, db2,
                 workspace, stream=None):
    b = saved if isinstance(saved, MoeBuffers) else buffers_struct(saved)
    _check("moe_backward", _lib.moe_backward(
        ctypes.byref(cfg), _ptr(x), _ptr(w_gate), _ptr(w1), _ptr(w2), ctypes.byref(b), _ptr(dy),
        _ptr(dx), _ptr(dw_gate), _ptr(dw1), _ptr(db1), _ptr(dw2), _ptr(db2), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_debug_set_wait_limit(ns: int):
    """Progress-wait limit of the single-launch gate kernel (0: 2 s)."""
    _check("moe_debug_set_wait_limit", _lib.moe_debug_set_wait_limit(int(ns)))


def moe_get_device_error() -> int:
    v = c_uint32()
    st = _lib.moe_get_device_error(ctypes.byref(v))
    if st not in (MOE_OK, MOE_ERR_DEVICE):
        raise MoeError("moe_get_device_error", st)
    return v.value
