"""Thin Python binding of libmoe's C ABI (include/moe.h).

Argument marshalling only: every function takes torch tensors (device memory
owned by the caller), passes their data pointers, the current CUDA stream and the
shape struct to the C entry point of the same name, and raises MoeError on a
non-zero status.  Every step of the layer runs in libmoe's kernels; if the
library is missing this module raises at import time instead of falling back to
anything else.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .synth import Workload

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_CHECK = 4, 5, 6
MOE_F32, MOE_BF16, MOE_MXFP8 = 0, 1, 2
DTYPES = {"f32": MOE_F32, "bf16": MOE_BF16, "mxfp8": MOE_MXFP8}

ENTRY_POINTS = (
    "moe_workspace_bytes", "moe_workspace_init", "moe_last_device_status", "moe_status_string",
    "moe_quantize_mxfp8", "moe_quantize_nvfp4", "moe_macro_workspace_bytes", "moe_forward_macrobatched",
    "moe_route_topk", "moe_layout", "moe_dispatch_pull", "moe_expert_ffn",
    "moe_combine", "moe_forward", "moe_forward_fused", "moe_min_minibatch", "moe_layout_noalloc",
    "moe_pack_expert_weights", "moe_backward_workspace_bytes", "moe_pack_expert_weights_dgrad",
    "moe_expert_ffn_train", "moe_forward_train", "moe_reverse_combine", "moe_expert_ffn_dgrad",
    "moe_reverse_dispatch", "moe_router_wgrad", "moe_backward", "moe_expert_wgrad",
)


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_name(status)} ({status})")


class Shape(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
                ("E", ctypes.c_int), ("k", ctypes.c_int), ("S", ctypes.c_int),
                ("dtype", ctypes.c_int)]

    @classmethod
    def of(cls, w: Workload) -> "Shape":
        return cls(w.N, w.H, w.I, w.E, w.k, w.S, DTYPES[w.dtype])


class Params(ctypes.Structure):
    _fields_ = [("ring_slots", ctypes.c_int), ("minibatch", ctypes.c_int),
                ("gather_ctas", ctypes.c_int), ("compute_ctas", ctypes.c_int),
                ("timeout_ns", ctypes.c_longlong), ("test_skip_ready", ctypes.c_int),
                ("reverse_ring", ctypes.c_int)]


class Saved(ctypes.Structure):
    """moe_saved_t: device pointers of the activations the backward reads."""
    _fields_ = [("idx", ctypes.c_void_p), ("gate", ctypes.c_void_p), ("inv", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p), ("sched", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("uv", ctypes.c_void_p)]

    @classmethod
    def of(cls, t: dict) -> "Saved":
        """From a dict of tensors with the field names as keys."""
        return cls(*(t[f].data_ptr() for f, _ in cls._fields_))


def load_library(path: str = _LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libmoe.so not built at {path}; run token_dispatch_expert_top_gb300.build")
    return ctypes.CDLL(path)


_lib = load_library()
_vp, _i, _i64, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
_shp, _prm, _svd = ctypes.POINTER(Shape), ctypes.POINTER(Params), ctypes.POINTER(Saved)
_SIGS = {
    "moe_workspace_bytes": (_sz, [_shp, _prm]),
    "moe_workspace_init": (_i, [_vp, _sz, _vp]),
    "moe_last_device_status": (_i, [_vp, _vp]),
    "moe_status_string": (ctypes.c_char_p, [_i]),
    "moe_quantize_mxfp8": (_i, [_vp, _i, _i64, _i64, _vp, _vp, _vp]),
    "moe_quantize_nvfp4": (_i, [_vp, _i, _i64, _i64, _vp, _vp, _vp, _vp]),
    "moe_macro_workspace_bytes": (_sz, [_shp, _prm, _i]),
    "moe_forward_macrobatched": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _shp, _prm, _i, _vp, _vp, _sz, _vp]),
    "moe_route_topk": (_i, [_vp, _vp, _vp, _shp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_layout": (_i, [_vp, _shp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_dispatch_pull": (_i, [_vp, _vp, _shp, _vp, _vp, _i, _i, _vp, _vp, _i, _vp, _sz, _vp]),
    "moe_expert_ffn": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _shp, _vp, _vp, _sz, _vp]),
    "moe_combine": (_i, [_vp, _vp, _vp, _shp, _vp, _vp, _sz, _vp]),
    "moe_forward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _shp, _prm, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_forward_fused": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _shp, _prm, _vp, _vp, _vp, _vp,
                               _sz, _vp]),
    "moe_min_minibatch": (_i, [_i, _i, _i, _i, _i]),
    "moe_layout_noalloc": (_i, [_vp, _shp, _vp, _vp, _vp, _vp, _vp]),
    "moe_pack_expert_weights": (_i, [_shp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "moe_backward_workspace_bytes": (_sz, [_shp]),
    "moe_pack_expert_weights_dgrad": (_i, [_shp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "moe_expert_ffn_train": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _shp, _vp, _vp, _vp, _sz, _vp]),
    "moe_forward_train": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _shp, _prm, _vp, _svd, _vp, _sz,
                               _vp]),
    "moe_reverse_combine": (_i, [_vp, _vp, _vp, _vp, _shp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                                 _vp]),
    "moe_expert_ffn_dgrad": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _shp, _vp, _vp, _vp, _vp,
                                  _vp, _sz, _vp]),
    "moe_reverse_dispatch": (_i, [_vp, _vp, _vp, _vp, _vp, _shp, _vp, _vp, _sz, _vp]),
    "moe_router_wgrad": (_i, [_vp, _vp, _vp, _vp, _shp, _vp, _vp, _vp, _sz, _vp]),
    "moe_backward": (_i, [_vp, _vp, _vp, _svd, _vp, _vp, _vp, _vp, _shp, _prm, _vp, _vp, _vp, _vp,
                          _vp, _vp, _sz, _vp]),
    "moe_expert_wgrad": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _shp, _vp, _vp, _vp, _sz, _vp]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def lib() -> ctypes.CDLL:
    return _lib


def status_name(code: int) -> str:
    return _lib.moe_status_string(code).decode()


def _p(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(fn: str, rc: int) -> None:
    if rc != MOE_OK:
        raise MoeError(fn, rc)


# ------------------------------------------------------------------ entry points
def moe_workspace_bytes(shape: Shape, params: Params | None = None) -> int:
    return _lib.moe_workspace_bytes(ctypes.byref(shape), ctypes.byref(params) if params else None)


def moe_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check("moe_workspace_init", _lib.moe_workspace_init(_p(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_last_device_status(ws: torch.Tensor, stream=None) -> int:
    return _lib.moe_last_device_status(_p(ws), _stream(stream))


def moe_status_string(code: int) -> str:
    return status_name(code)


def moe_quantize_mxfp8(inp: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, stream=None) -> None:
    dt = MOE_BF16 if inp.dtype == torch.bfloat16 else MOE_F32
    K = inp.shape[-1]
    rows = inp.numel() // K
    _check("moe_quantize_mxfp8", _lib.moe_quantize_mxfp8(_p(inp), dt, rows, K, _p(codes), _p(scales),
                                                         _stream(stream)))


def moe_quantize_nvfp4(inp: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor,
                       tensor_scale: torch.Tensor, stream=None) -> None:
    dt = MOE_BF16 if inp.dtype == torch.bfloat16 else MOE_F32
    K = inp.shape[-1]
    rows = inp.numel() // K
    _check("moe_quantize_nvfp4", _lib.moe_quantize_nvfp4(_p(inp), dt, rows, K, _p(codes), _p(scales),
                                                         _p(tensor_scale), _stream(stream)))


def moe_pack_expert_weights(shape: Shape, w_gate_up, w_gu_scales, w_down, w_d_scales,
                            packed_gate_up, packed_gu_scales, packed_down, packed_d_scales,
                            stream=None) -> None:
    _check("moe_pack_expert_weights", _lib.moe_pack_expert_weights(
        ctypes.byref(shape), _p(w_gate_up), _p(w_gu_scales), _p(w_down), _p(w_d_scales),
        _p(packed_gate_up), _p(packed_gu_scales), _p(packed_down), _p(packed_d_scales),
        _stream(stream)))


def _wsz(ws):
    return 0 if ws is None else ws.numel() * ws.element_size()


def moe_route_topk(x, w_router, bias, shape: Shape, idx, gate, logits_out=None, xq_codes=None,
                   xq_scales=None, ws=None, stream=None) -> None:
    _check("moe_route_topk", _lib.moe_route_topk(
        _p(x), _p(w_router), _p(bias), ctypes.byref(shape), _p(idx), _p(gate), _p(logits_out),
        _p(xq_codes), _p(xq_scales), _p(ws), _wsz(ws), _stream(stream)))


def moe_layout(idx, shape: Shape, counts, offsets, sched, inv, ws, stream=None) -> None:
    _check("moe_layout", _lib.moe_layout(_p(idx), ctypes.byref(shape), _p(counts), _p(offsets),
                                         _p(sched), _p(inv), _p(ws), _wsz(ws), _stream(stream)))


def moe_dispatch_pull(shard_rows, shard_scales, shape: Shape, sched, inv, slot_begin: int,
                      slot_count: int, ring, ring_scales, ring_slots: int, ws, stream=None) -> None:
    """shard_rows / shard_scales: int64 device tensors holding S device pointers;
    inv: the [N][k] inverse map (visit slots token by token) or None (slot order)."""
    _check("moe_dispatch_pull", _lib.moe_dispatch_pull(
        _p(shard_rows), _p(shard_scales), ctypes.byref(shape), _p(sched), _p(inv), slot_begin,
        slot_count, _p(ring), _p(ring_scales), ring_slots, _p(ws), _wsz(ws), _stream(stream)))


def moe_expert_ffn(a, a_scales, offsets, w_gate_up, w_gu_scales, w_down, w_d_scales, shape: Shape,
                   y, ws, stream=None) -> None:
    _check("moe_expert_ffn", _lib.moe_expert_ffn(
        _p(a), _p(a_scales), _p(offsets), _p(w_gate_up), _p(w_gu_scales), _p(w_down),
        _p(w_d_scales), ctypes.byref(shape), _p(y), _p(ws), _wsz(ws), _stream(stream)))


def moe_combine(y, inv, gate, shape: Shape, out, ws, stream=None) -> None:
    _check("moe_combine", _lib.moe_combine(_p(y), _p(inv), _p(gate), ctypes.byref(shape), _p(out),
                                           _p(ws), _wsz(ws), _stream(stream)))


def moe_forward(x, w_router, bias, w_gate_up, w_gu_scales, w_down, w_d_scales, shape: Shape,
                params: Params | None, out, idx_out, gate_out, ws, stream=None) -> None:
    _check("moe_forward", _lib.moe_forward(
        _p(x), _p(w_router), _p(bias), _p(w_gate_up), _p(w_gu_scales), _p(w_down), _p(w_d_scales),
        ctypes.byref(shape), ctypes.byref(params) if params else None, _p(out), _p(idx_out),
        _p(gate_out), _p(ws), _wsz(ws), _stream(stream)))


def moe_macro_workspace_bytes(shape: Shape, params: Params | None, macrobatches: int) -> int:
    return _lib.moe_macro_workspace_bytes(ctypes.byref(shape), ctypes.byref(params) if params else None,
                                          macrobatches)


def moe_forward_macrobatched(x, w_router, bias, w_gate_up, w_gu_scales, w_down, w_d_scales, shape: Shape,
                             params: Params | None, macrobatches: int, out, ws, stream=None) -> None:
    _check("moe_forward_macrobatched", _lib.moe_forward_macrobatched(
        _p(x), _p(w_router), _p(bias), _p(w_gate_up), _p(w_gu_scales), _p(w_down), _p(w_d_scales),
        ctypes.byref(shape), ctypes.byref(params) if params else None, macrobatches, _p(out), _p(ws),
        _wsz(ws), _stream(stream)))


def moe_forward_fused(x, w_router, bias, w_gate_up, w_gu_scales, w_down, w_d_scales, shape: Shape,
                      params: Params | None, out, idx_out, gate_out, ws, stream=None) -> None:
    _check("moe_forward_fused", _lib.moe_forward_fused(
        _p(x), _p(w_router), _p(bias), _p(w_gate_up), _p(w_gu_scales), _p(w_down), _p(w_d_scales),
        ctypes.byref(shape), ctypes.byref(params) if params else None, _p(out), _p(idx_out),
        _p(gate_out), _p(ws), _wsz(ws), _stream(stream)))


def moe_min_minibatch(waves: int, compute_sms: int, tile_m: int, tile_n: int, I: int) -> int:
    return _lib.moe_min_minibatch(waves, compute_sms, tile_m, tile_n, I)


def moe_layout_noalloc(idx, shape: Shape, counts, offsets, sched, inv, stream=None) -> None:
    """moe_layout for callers that cannot allocate: no workspace argument; the
    library's fixed device scratch array is used instead (see include/moe.h)."""
    _check("moe_layout_noalloc", _lib.moe_layout_noalloc(
        _p(idx), ctypes.byref(shape), _p(counts), _p(offsets), _p(sched), _p(inv), _stream(stream)))


# ------------------------------------------------------------------ backward
def moe_backward_workspace_bytes(shape: Shape) -> int:
    return _lib.moe_backward_workspace_bytes(ctypes.byref(shape))


def moe_pack_expert_weights_dgrad(shape: Shape, w_gate_up, w_down, packed_gate_up_t,
                                  packed_gu_t_scales, packed_down_t, packed_d_t_scales,
                                  stream=None) -> None:
    _check("moe_pack_expert_weights_dgrad", _lib.moe_pack_expert_weights_dgrad(
        ctypes.byref(shape), _p(w_gate_up), _p(w_down), _p(packed_gate_up_t),
        _p(packed_gu_t_scales), _p(packed_down_t), _p(packed_d_t_scales), _stream(stream)))


def moe_expert_ffn_train(a, a_scales, offsets, w_gate_up, w_gu_scales, w_down, w_d_scales,
                         shape: Shape, y, uv, ws, stream=None) -> None:
    _check("moe_expert_ffn_train", _lib.moe_expert_ffn_train(
        _p(a), _p(a_scales), _p(offsets), _p(w_gate_up), _p(w_gu_scales), _p(w_down),
        _p(w_d_scales), ctypes.byref(shape), _p(y), _p(uv), _p(ws), _wsz(ws), _stream(stream)))


def moe_forward_train(x, w_router, bias, w_gate_up, w_gu_scales, w_down, w_d_scales,
                      shape: Shape, params: Params | None, out, saved: Saved, ws,
                      stream=None) -> None:
    _check("moe_forward_train", _lib.moe_forward_train(
        _p(x), _p(w_router), _p(bias), _p(w_gate_up), _p(w_gu_scales), _p(w_down), _p(w_d_scales),
        ctypes.byref(shape), ctypes.byref(params) if params else None, _p(out),
        ctypes.byref(saved), _p(ws), _wsz(ws), _stream(stream)))


def moe_reverse_combine(dout, y, inv, gate, shape: Shape, dy, dy_scales, dgate, dlogit,
                        slot_gate, slot_dlogit, ws, stream=None) -> None:
    _check("moe_reverse_combine", _lib.moe_reverse_combine(
        _p(dout), _p(y), _p(inv), _p(gate), ctypes.byref(shape), _p(dy), _p(dy_scales),
        _p(dgate), _p(dlogit), _p(slot_gate), _p(slot_dlogit), _p(ws), _wsz(ws), _stream(stream)))


def moe_expert_ffn_dgrad(dy, dy_scales, uv, offsets, wt_gate_up, wt_gu_scales, wt_down,
                         wt_d_scales, shape: Shape, duv, duv_codes, duv_scales, da, ws,
                         stream=None) -> None:
    _check("moe_expert_ffn_dgrad", _lib.moe_expert_ffn_dgrad(
        _p(dy), _p(dy_scales), _p(uv), _p(offsets), _p(wt_gate_up), _p(wt_gu_scales),
        _p(wt_down), _p(wt_d_scales), ctypes.byref(shape), _p(duv), _p(duv_codes),
        _p(duv_scales), _p(da), _p(ws), _wsz(ws), _stream(stream)))


def moe_reverse_dispatch(da, inv, idx, dlogit, w_router, shape: Shape, dx, ws, stream=None) -> None:
    _check("moe_reverse_dispatch", _lib.moe_reverse_dispatch(
        _p(da), _p(inv), _p(idx), _p(dlogit), _p(w_router), ctypes.byref(shape), _p(dx), _p(ws),
        _wsz(ws), _stream(stream)))


def moe_router_wgrad(x, sched, offsets, slot_dlogit, shape: Shape, dw_router, dbias, ws,
                     stream=None) -> None:
    _check("moe_router_wgrad", _lib.moe_router_wgrad(
        _p(x), _p(sched), _p(offsets), _p(slot_dlogit), ctypes.byref(shape), _p(dw_router),
        _p(dbias), _p(ws), _wsz(ws), _stream(stream)))


def moe_expert_wgrad(duv, x, dout, uv, sched, slot_gate, offsets, shape: Shape, dw_gate_up, dw_down,
                     ws, stream=None) -> None:
    _check("moe_expert_wgrad", _lib.moe_expert_wgrad(
        _p(duv), _p(x), _p(dout), _p(uv), _p(sched), _p(slot_gate), _p(offsets),
        ctypes.byref(shape), _p(dw_gate_up), _p(dw_down), _p(ws), _wsz(ws), _stream(stream)))


def moe_backward(dout, x, w_router, saved: Saved, wt_gate_up, wt_gu_scales, wt_down, wt_d_scales,
                 shape: Shape, params: Params | None, dx, dw_router, dbias, dw_gate_up, dw_down, ws,
                 stream=None) -> None:
    _check("moe_backward", _lib.moe_backward(
        _p(dout), _p(x), _p(w_router), ctypes.byref(saved), _p(wt_gate_up), _p(wt_gu_scales),
        _p(wt_down), _p(wt_d_scales), ctypes.byref(shape), ctypes.byref(params) if params else None,
        _p(dx), _p(dw_router), _p(dbias), _p(dw_gate_up), _p(dw_down), _p(ws), _wsz(ws),
        _stream(stream)))
