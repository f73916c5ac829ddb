"""GB300 (sm_103a) routed-expert FP4 MoE layer: Python binding of the C-ABI library.

The functions below carry the names of the C entry points in include/fp4moe.h and only
marshal arguments (torch tensors -> device pointers, the current CUDA stream).  Every step
of the layer runs in the library's CUDA kernels; there is no CPU or PyTorch fallback: if
the shared library is missing, importing the binding raises.

Tensor conventions: bf16 tensors may be torch.bfloat16 or int16/uint16 bit patterns; all
tensors must be contiguous CUDA tensors on the current device.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

__all__ = [
    "MoeError", "moe_dims", "moe_arena", "lib", "moe_slot_bytes", "moe_workspace_bytes",
    "moe_workspace_init", "moe_pack_expert", "moe_route_topk", "moe_route_topk_noalloc", "moe_permute",
    "moe_expert_ffn_fp4", "moe_layer_decode_fp4", "moe_combine", "moe_residency_bias", "moe_split_waves", "moe_gather_experts", "moe_status_str",
    "moe_cb3_slot_bytes", "moe_pack_cb3", "moe_expert_ffn_cb3", "moe_expert_ffn_cb3_rows", "MOE_STATUS_CB3_ROW",
    "moe_kernel_launches", "moe_workspace_set_wait_limit", "moe_residual_rmsnorm", "MOE_FUSE_COMBINE", "MOE_FFN_CUDA_CORES",
    "MOE_STATUS_FEW_RESIDENT", "MOE_STATUS_BAD_SLOT", "MOE_STATUS_TIMEOUT", "DECODE_MAX_T",
]

MOE_FUSE_COMBINE = 1
MOE_FFN_CUDA_CORES = 2
MOE_STATUS_FEW_RESIDENT = 1
MOE_STATUS_BAD_SLOT = 2
MOE_STATUS_TIMEOUT = 4
MOE_STATUS_CB3_ROW = 8
DECODE_MAX_T = 16


class moe_dims(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("f", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32)]


class moe_arena(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("slot_bytes", ctypes.c_int64), ("num_slots", ctypes.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int, text: str):
        super().__init__("%s failed: %d (%s)" % (fn, code, text))
        self.code = code


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int32
_SIG = {
    "moe_slot_bytes": (ctypes.c_int64, [_P]),
    "moe_workspace_bytes": (ctypes.c_size_t, [_P, _I]),
    "moe_workspace_init": (ctypes.c_int, [_P, _P, ctypes.c_size_t, _P]),
    "moe_workspace_set_wait_limit": (ctypes.c_int, [_P, _P, ctypes.c_size_t, _I, _P]),
    "moe_pack_expert": (ctypes.c_int, [_P] * 8 + [_I, _P]),
    "moe_route_topk": (ctypes.c_int, [_P, _I] + [_P] * 9 + [ctypes.c_size_t, _P]),
    "moe_permute": (ctypes.c_int, [_P, _I] + [_P] * 5 + [ctypes.c_size_t, _P]),
    "moe_expert_ffn_fp4": (ctypes.c_int, [_P, _P, _I] + [_P] * 7 + [_I] + [_P] * 4 + [ctypes.c_size_t, _P]),
    "moe_layer_decode_fp4": (ctypes.c_int, [_P, _P, _I] + [_P] * 10 + [ctypes.c_size_t, _P]),
    "moe_combine": (ctypes.c_int, [_P, _I] + [_P] * 5),
    "moe_residency_bias": (ctypes.c_int, [_P, _P, _P, _P, _I, ctypes.c_float, _P, _P]),
    "moe_cb3_slot_bytes": (ctypes.c_int64, [_P]),
    "moe_pack_cb3": (ctypes.c_int, [_P, _P, _I, _P, _I, _P, _P]),
    "moe_expert_ffn_cb3": (ctypes.c_int, [_P, _P, _I] + [_P] * 6 + [ctypes.c_size_t, _P]),
    "moe_expert_ffn_cb3_rows": (ctypes.c_int, [_P, _P, _I] + [_P] * 6 + [ctypes.c_size_t, _P]),
    "moe_split_waves": (ctypes.c_int, [_P, _I, _P, _P, _P, _I, _P, _P, _P, _P, _P]),
    "moe_gather_experts": (ctypes.c_int, [_P, _P, _P, _I] + [_P] * 6),
    "moe_route_topk_noalloc": (ctypes.c_int, [_P, _I] + [_P] * 9),
    "moe_residual_rmsnorm": (ctypes.c_int, [_I, _I, _P, _P, ctypes.c_float, _P, _P]),
    "moe_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_kernel_launches": (ctypes.c_uint64, []),
}


def lib(path: str | None = None):
    """Load (building first if needed) the CUDA library; raises if it cannot be loaded."""
    global _lib
    if _lib is None:
        p = path or _build.LIB
        if not os.path.exists(p):
            p = _build.build()
        L = ctypes.CDLL(p)
        for name, (res, args) in _SIG.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, rc: int):
    if rc != 0:
        raise MoeError(fn, rc, moe_status_str(rc))
    return rc


def _dims(d):
    return d if isinstance(d, moe_dims) else moe_dims(*d)


def moe_status_str(code: int) -> str:
    return lib().moe_status_str(int(code)).decode()


def moe_kernel_launches() -> int:
    """Kernels the library has enqueued in this process (a graph capture counts once)."""
    return int(lib().moe_kernel_launches())


def moe_slot_bytes(dims) -> int:
    return int(lib().moe_slot_bytes(ctypes.byref(_dims(dims))))


def moe_workspace_bytes(dims, T_max: int) -> int:
    return int(lib().moe_workspace_bytes(ctypes.byref(_dims(dims)), int(T_max)))


def moe_workspace_init(dims, ws, stream=None):
    _check("moe_workspace_init", lib().moe_workspace_init(ctypes.byref(_dims(dims)), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_workspace_set_wait_limit(dims, ws, polls: int, stream=None):
    """Diagnostic: dependency waits of the expert kernels on this workspace give up after
    `polls` polls (0 restores the default)."""
    _check("moe_workspace_set_wait_limit", lib().moe_workspace_set_wait_limit(
        ctypes.byref(_dims(dims)), _ptr(ws), ws.numel() * ws.element_size(), int(polls), _stream(stream)))


def moe_pack_expert(dims, gate_q, gate_s, up_q, up_s, down_q, down_s, arena: moe_arena, slot: int, stream=None):
    _check("moe_pack_expert", lib().moe_pack_expert(
        ctypes.byref(_dims(dims)), _ptr(gate_q), _ptr(gate_s), _ptr(up_q), _ptr(up_s), _ptr(down_q), _ptr(down_s),
        ctypes.byref(arena), int(slot), _stream(stream)))


def moe_route_topk(dims, T, x, w_router, score_bias, expert_to_slot, topk_ids, topk_w, topk_slot, dev_status,
                   ws, stream=None):
    _check("moe_route_topk", lib().moe_route_topk(
        ctypes.byref(_dims(dims)), int(T), _ptr(x), _ptr(w_router), _ptr(score_bias), _ptr(expert_to_slot),
        _ptr(topk_ids), _ptr(topk_w), _ptr(topk_slot), _ptr(dev_status), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def moe_route_topk_noalloc(dims, T, x, w_router, score_bias, expert_to_slot, topk_ids, topk_w, topk_slot,
                           dev_status, stream=None):
    """moe_route_topk with the library's own static scratch (no workspace; T <= 16)."""
    _check("moe_route_topk_noalloc", lib().moe_route_topk_noalloc(
        ctypes.byref(_dims(dims)), int(T), _ptr(x), _ptr(w_router), _ptr(score_bias), _ptr(expert_to_slot),
        _ptr(topk_ids), _ptr(topk_w), _ptr(topk_slot), _ptr(dev_status), _stream(stream)))


def moe_permute(dims, T, topk_ids, group_offsets, row_src, row_dst, ws, stream=None):
    _check("moe_permute", lib().moe_permute(
        ctypes.byref(_dims(dims)), int(T), _ptr(topk_ids), _ptr(group_offsets), _ptr(row_src), _ptr(row_dst),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_expert_ffn_fp4(dims, arena: moe_arena, T, x, topk_ids, topk_slot, topk_w, group_offsets, row_src, row_dst,
                       flags, rows_out, y, dev_status, ws, stream=None):
    _check("moe_expert_ffn_fp4", lib().moe_expert_ffn_fp4(
        ctypes.byref(_dims(dims)), ctypes.byref(arena), int(T), _ptr(x), _ptr(topk_ids), _ptr(topk_slot),
        _ptr(topk_w), _ptr(group_offsets), _ptr(row_src), _ptr(row_dst), int(flags), _ptr(rows_out), _ptr(y),
        _ptr(dev_status), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_layer_decode_fp4(dims, arena: moe_arena, T, x, w_router, score_bias, expert_to_slot, topk_ids, topk_w,
                         topk_slot, y, dev_status, ws, stream=None):
    _check("moe_layer_decode_fp4", lib().moe_layer_decode_fp4(
        ctypes.byref(_dims(dims)), ctypes.byref(arena), int(T), _ptr(x), _ptr(w_router), _ptr(score_bias),
        _ptr(expert_to_slot), _ptr(topk_ids), _ptr(topk_w), _ptr(topk_slot), _ptr(y), _ptr(dev_status), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def moe_residual_rmsnorm(T, d, x, y, eps, x_next, stream=None):
    """x_next = bf16(RMSNorm(x + y)) (unit weight), the chaining step of multi-layer workloads."""
    _check("moe_residual_rmsnorm", lib().moe_residual_rmsnorm(int(T), int(d), _ptr(x), _ptr(y), ctypes.c_float(eps),
                                                              _ptr(x_next), _stream(stream)))


def moe_combine(dims, T, rows, row_dst, topk_w, y, stream=None):
    _check("moe_combine", lib().moe_combine(
        ctypes.byref(_dims(dims)), int(T), _ptr(rows), _ptr(row_dst), _ptr(topk_w), _ptr(y), _stream(stream)))


def moe_residency_bias(dims, score_bias, expert_to_slot, resident_expert, num_slots, lam, bias_out, stream=None):
    _check("moe_residency_bias", lib().moe_residency_bias(
        ctypes.byref(_dims(dims)), _ptr(score_bias), _ptr(expert_to_slot), _ptr(resident_expert), int(num_slots),
        float(lam), _ptr(bias_out), _stream(stream)))


def moe_cb3_slot_bytes(dims) -> int:
    return int(lib().moe_cb3_slot_bytes(ctypes.byref(_dims(dims))))


def moe_pack_cb3(dims, fp4_arena, fp4_slot, cb3_arena, cb3_slot, status, stream=None):
    _check("moe_pack_cb3", lib().moe_pack_cb3(ctypes.byref(_dims(dims)), ctypes.byref(fp4_arena), int(fp4_slot),
                                              ctypes.byref(cb3_arena), int(cb3_slot), _ptr(status), _stream(stream)))


def moe_expert_ffn_cb3(dims, cb3_arena, T, x, topk_slot, topk_w, y, status, ws, stream=None):
    _check("moe_expert_ffn_cb3", lib().moe_expert_ffn_cb3(
        ctypes.byref(_dims(dims)), ctypes.byref(cb3_arena), int(T), _ptr(x), _ptr(topk_slot), _ptr(topk_w), _ptr(y),
        _ptr(status), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_expert_ffn_cb3_rows(dims, cb3_arena, T, x, topk_slot, row_dst, rows_out, status, ws, stream=None):
    """moe_expert_ffn_cb3 without the combine: pair (t, j) into row row_dst[t*k + j] of rows_out."""
    _check("moe_expert_ffn_cb3_rows", lib().moe_expert_ffn_cb3_rows(
        ctypes.byref(_dims(dims)), ctypes.byref(cb3_arena), int(T), _ptr(x), _ptr(topk_slot), _ptr(row_dst),
        _ptr(rows_out), _ptr(status), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_split_waves(dims, T, topk_ids, topk_slot, resident_expert, num_slots, slot_wave1, slot_wave2, missing,
                    n_missing, stream=None):
    _check("moe_split_waves", lib().moe_split_waves(
        ctypes.byref(_dims(dims)), int(T), _ptr(topk_ids), _ptr(topk_slot), _ptr(resident_expert), int(num_slots),
        _ptr(slot_wave1), _ptr(slot_wave2), _ptr(missing), _ptr(n_missing), _stream(stream)))


def moe_gather_experts(dims, arena, store_ptr, n_store, missing, n_missing, expert_to_slot, resident_expert,
                       dev_status, stream=None):
    """store_ptr: int device-accessible address of the slot images (device memory, or pinned
    host memory mapped into the device)."""
    _check("moe_gather_experts", lib().moe_gather_experts(
        ctypes.byref(_dims(dims)), ctypes.byref(arena), ctypes.c_void_p(int(store_ptr)), int(n_store), _ptr(missing),
        _ptr(n_missing), _ptr(expert_to_slot), _ptr(resident_expert), _ptr(dev_status), _stream(stream)))


from .layer import MoeLayer  # noqa: E402  (device buffers + the four calls in order)

__all__.append("MoeLayer")
