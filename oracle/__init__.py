"""CPU oracle for the routed-expert FP4 MoE layer -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  It wraps ``moe_oracle.c`` (plain single-threaded C) through ctypes
and shares nothing with the CUDA library.  Functions take and return numpy arrays; bf16
tensors are passed as uint16 bit patterns.

Parity status per function (what pins it is in tests/test_oracle_pins.py):
  e2m1 / UE8M0 / bf16 decoding   pinned (bit-field definitions, library conversions)
  exact fp32 router logit        pinned (exact rational arithmetic, hand-made midpoints)
  router score                   pinned (multi-precision sigmoid, special values)
  route_topk                     pinned (hand-worked examples in tests/golden/)
  residency_bias                 pinned (hand-worked values, brute-force routing limits)
  cb3_pack_row / cb3_expert_ffn  pinned (exhaustive partitions in exact rationals, lossless
                                 rows, FP4 FFN on lossless experts)
  permute                        pinned (brute force and invariants)
  expert_ffn_f32 / combine_f32   pinned (fp32 closed forms with exact sums, an independent
    / layer (fp32, the reference)  numpy float32 sequential re-derivation, agreement with the
                                 fp64 statement within the fp32 summation bound)
  expert_ffn / combine (fp64)    pinned (closed forms, independent fp64 re-derivation); kept as
                                 a cross-check of the fp32 statement
  residual_rmsnorm               pinned (independent fp64 re-derivation)
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32 = ctypes.c_int
        L.oracle_e2m1_value.restype = ctypes.c_double
        L.oracle_e2m1_value.argtypes = [i32]
        L.oracle_ue8m0_value.restype = ctypes.c_double
        L.oracle_ue8m0_value.argtypes = [i32]
        L.oracle_bf16_value.restype = ctypes.c_double
        L.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_from_double.restype = ctypes.c_uint16
        L.oracle_bf16_from_double.argtypes = [ctypes.c_double]
        L.oracle_code_at.restype = i32
        L.oracle_code_at.argtypes = [P, i32]
        L.oracle_weight_at.restype = ctypes.c_double
        L.oracle_weight_at.argtypes = [P, P, i32]
        L.oracle_dot_bf16_rn32.restype = ctypes.c_float
        L.oracle_dot_bf16_rn32.argtypes = [P, P, i32, P]
        L.oracle_router_score.restype = ctypes.c_float
        L.oracle_router_score.argtypes = [ctypes.c_float]
        L.oracle_residency_bias.restype = None
        L.oracle_residency_bias.argtypes = [i32, P, P, P, i32, ctypes.c_float, P]
        L.oracle_cb3_pack_row.restype = i32
        L.oracle_cb3_pack_row.argtypes = [i32, P, P, P, P]
        L.oracle_cb3_pack_matrix.restype = None
        L.oracle_cb3_pack_matrix.argtypes = [i32, i32, P, P, P, P]
        L.oracle_cb3_expert_ffn.restype = None
        L.oracle_cb3_expert_ffn.argtypes = [i32, i32] + [P] * 9
        L.oracle_route_topk.restype = i32
        L.oracle_route_topk.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P, P, P]
        L.oracle_permute.restype = i32
        L.oracle_permute.argtypes = [i32, i32, i32, P, P, P, P]
        L.oracle_expert_ffn.restype = None
        L.oracle_expert_ffn.argtypes = [i32, i32, P, P, P, P, P, P, P, P, P]
        L.oracle_combine.restype = None
        L.oracle_combine.argtypes = [i32, i32, P, P, P]
        L.oracle_expert_ffn_f32.restype = None
        L.oracle_expert_ffn_f32.argtypes = [i32, i32, P, P, P, P, P, P, P, P, P]
        L.oracle_combine_f32.restype = None
        L.oracle_combine_f32.argtypes = [i32, i32, P, P, P]
        L.oracle_weight_at_f32.restype = ctypes.c_float
        L.oracle_weight_at_f32.argtypes = [P, P, i32]
        L.oracle_moe_layer_f32.restype = i32
        L.oracle_moe_layer_f32.argtypes = [i32] * 6 + [P] * 15
        L.oracle_moe_layer.restype = i32
        L.oracle_moe_layer.argtypes = [i32] * 6 + [P] * 15
        L.oracle_residual_rmsnorm.restype = None
        L.oracle_residual_rmsnorm.argtypes = [i32, i32, P, P, ctypes.c_double, P]
        L.oracle_expert_bytes.restype = ctypes.c_longlong
        L.oracle_expert_bytes.argtypes = [i32, i32]
        _lib = L
    return _lib


def _c(a, dtype):
    """Contiguous array of the given dtype (kept alive by the caller)."""
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(int(code))


def ue8m0_value(byte: int) -> float:
    return lib().oracle_ue8m0_value(int(byte))


def bf16_value(bits: int) -> float:
    return lib().oracle_bf16_value(int(bits))


def bf16_from_double(v: float) -> int:
    return int(lib().oracle_bf16_from_double(float(v)))


def dot_bf16_rn32(x_bits, w_bits):
    x = _c(x_bits, np.uint16)
    w = _c(w_bits, np.uint16)
    bad = ctypes.c_int(0)
    v = lib().oracle_dot_bf16_rn32(_p(x), _p(w), int(x.size), ctypes.byref(bad))
    return np.float32(v), bool(bad.value)


def router_score(logit) -> np.float32:
    return np.float32(lib().oracle_router_score(float(np.float32(logit))))


def route_topk(x_bits, w_router_bits, bias, expert_to_slot, k, want_logits=False):
    """Returns dict(ids, weights, slots, status[, logits, scores])."""
    x = _c(x_bits, np.uint16)
    wr = _c(w_router_bits, np.uint16)
    T, d = x.shape
    E = wr.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    tab = _c(expert_to_slot, np.int32)
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    slots = np.zeros((T, k), np.int32)
    lg = np.zeros((T, E), np.float32) if want_logits else None
    sc = np.zeros((T, E), np.float32) if want_logits else None
    st = lib().oracle_route_topk(T, d, E, k, _p(x), _p(wr), _p(b), _p(tab), _p(ids), _p(w),
                                 _p(slots), _p(lg), _p(sc))
    out = dict(ids=ids, weights=w, slots=slots, status=int(st))
    if want_logits:
        out["logits"], out["scores"] = lg, sc
    return out


def residency_bias(bias, expert_to_slot, resident_expert, lam):
    """Cache-conditional routing bias: bias + lam (fp32) for experts resident in their slot."""
    tab = _c(expert_to_slot, np.int32)
    res = _c(resident_expert, np.int32)
    b = None if bias is None else _c(bias, np.float32)
    out = np.zeros(tab.shape[0], np.float32)
    lib().oracle_residency_bias(tab.shape[0], _p(b), _p(tab), _p(res), res.shape[0], ctypes.c_float(lam), _p(out))
    return out


def permute(ids, E):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    offsets = np.zeros(E + 1, np.int32)
    row_src = np.full(T * k, -1, np.int32)
    row_dst = np.full(T * k, -1, np.int32)
    n = lib().oracle_permute(T, k, E, _p(ids), _p(offsets), _p(row_src), _p(row_dst))
    return dict(offsets=offsets, row_src=row_src[:n].copy(), row_dst=row_dst, rows=int(n))


def expert_ffn_f32(x_bits, ex: dict):
    """One expert on one token in fp32, every sum in index order (the reference statement);
    returns (h [f], z [d]) as float32."""
    x = _c(x_bits, np.uint16)
    d = x.size
    gq = _c(ex["gate_q"], np.uint8)
    f = gq.shape[0]
    arrs = [gq] + [_c(ex[n], np.uint8) for n in ("gate_s", "up_q", "up_s", "down_q", "down_s")]
    h = np.zeros(f, np.float32)
    z = np.zeros(d, np.float32)
    lib().oracle_expert_ffn_f32(d, f, _p(x), *[_p(a) for a in arrs], _p(h), _p(z))
    return h, z


def combine_f32(z, w):
    """y = sum_j w_j z_j in fp32, j ascending."""
    z = _c(z, np.float32)
    w = _c(w, np.float32)
    k, d = z.shape
    y = np.zeros(d, np.float32)
    lib().oracle_combine_f32(d, k, _p(z), _p(w), _p(y))
    return y


def weight_at_f32(q_row, s_row, k: int) -> np.float32:
    q = _c(q_row, np.uint8)
    sc = _c(s_row, np.uint8)
    return np.float32(lib().oracle_weight_at_f32(_p(q), _p(sc), int(k)))


def expert_ffn(x_bits, ex: dict):
    """One expert (canonical tensors dict) on one token; returns (h [f], z [d]) in fp64
    (the cross-check statement; expert_ffn_f32 is the reference)."""
    x = _c(x_bits, np.uint16)
    d = x.size
    gq = _c(ex["gate_q"], np.uint8)
    f = gq.shape[0]
    arrs = [gq] + [_c(ex[n], np.uint8) for n in ("gate_s", "up_q", "up_s", "down_q", "down_s")]
    h = np.zeros(f, np.float64)
    z = np.zeros(d, np.float64)
    lib().oracle_expert_ffn(d, f, _p(x), *[_p(a) for a in arrs], _p(h), _p(z))
    return h, z


def cb3_pack_row(q_row, s_row):
    """One FP4 row (packed codes, UE8M0 scales) -> (levels uint16 bf16 bits [8], idx uint8 [K],
    number of distinct values)."""
    q = _c(q_row, np.uint8)
    sc = _c(s_row, np.uint8)
    K = q.size * 2
    cb = np.zeros(8, np.uint16)
    idx = np.zeros(K, np.uint8)
    n = lib().oracle_cb3_pack_row(K, _p(q), _p(sc), _p(cb), _p(idx))
    return cb, idx, int(n)


def cb3_pack_expert(ex: dict):
    """Canonical FP4 expert tensors -> dict of cb3 levels [rows, 8] and indices [rows, K] for
    the gate, up and down matrices."""
    out = {}
    for m in ("gate", "up", "down"):
        q, sc = _c(ex[m + "_q"], np.uint8), _c(ex[m + "_s"], np.uint8)
        R, K = q.shape[0], q.shape[1] * 2
        cb = np.zeros((R, 8), np.uint16)
        idx = np.zeros((R, K), np.uint8)
        lib().oracle_cb3_pack_matrix(R, K, _p(q), _p(sc), _p(cb), _p(idx))
        out[m + "_cb"], out[m + "_idx"] = cb, idx
    return out


def cb3_expert_ffn(x_bits, cx: dict):
    """One cb3 expert (cb3_pack_expert's dict) on one token; returns (h [f], z [d]) in fp64."""
    x = _c(x_bits, np.uint16)
    d = x.size
    f = cx["gate_cb"].shape[0]
    arrs = []
    for m in ("gate", "up", "down"):
        arrs += [_c(cx[m + "_cb"], np.uint16), _c(cx[m + "_idx"], np.uint8)]
    h = np.zeros(f, np.float64)
    z = np.zeros(d, np.float64)
    lib().oracle_cb3_expert_ffn(d, f, _p(x), *[_p(a) for a in arrs], _p(h), _p(z))
    return h, z


def combine(z, w):
    z = _c(z, np.float64)
    w = _c(w, np.float32)
    k, d = z.shape
    y = np.zeros(d, np.float64)
    lib().oracle_combine(d, k, _p(z), _p(w), _p(y))
    return y


def moe_layer(x_bits, w_router_bits, bias, expert_to_slot, k, slot_tensors: dict, precision: str = "f32"):
    """Whole layer with every slot's canonical tensors stacked as [num_slots, ...].
    precision "f32" (the reference statement) or "f64" (the cross-check); y is returned as
    float64 either way (exact conversion of the fp32 result)."""
    x = _c(x_bits, np.uint16)
    wr = _c(w_router_bits, np.uint16)
    T, d = x.shape
    E = wr.shape[0]
    gq = _c(slot_tensors["gate_q"], np.uint8)
    S, f = gq.shape[0], gq.shape[1]
    arrs = [gq] + [_c(slot_tensors[n], np.uint8) for n in ("gate_s", "up_q", "up_s", "down_q", "down_s")]
    b = None if bias is None else _c(bias, np.float32)
    tab = _c(expert_to_slot, np.int32)
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    slots = np.zeros((T, k), np.int32)
    yb = np.zeros((T, d), np.uint16)
    if precision == "f32":
        y = np.zeros((T, d), np.float32)
        st = lib().oracle_moe_layer_f32(T, d, f, E, k, S, _p(x), _p(wr), _p(b), _p(tab),
                                        *[_p(a) for a in arrs], _p(ids), _p(w), _p(slots), _p(y), _p(yb))
        y = y.astype(np.float64)
    elif precision == "f64":
        y = np.zeros((T, d), np.float64)
        st = lib().oracle_moe_layer(T, d, f, E, k, S, _p(x), _p(wr), _p(b), _p(tab),
                                    *[_p(a) for a in arrs], _p(ids), _p(w), _p(slots), _p(y), _p(yb))
    else:
        raise ValueError("precision must be 'f32' or 'f64'")
    return dict(ids=ids, weights=w, slots=slots, y=y, y_bf16=yb, status=int(st))


def residual_rmsnorm(x_bits, y, eps=1e-6):
    x = _c(x_bits, np.uint16)
    y = _c(y, np.float64)
    T, d = x.shape
    out = np.zeros((T, d), np.uint16)
    lib().oracle_residual_rmsnorm(T, d, _p(x), _p(y), float(eps), _p(out))
    return out


def expert_bytes(d: int, f: int) -> int:
    return int(lib().oracle_expert_bytes(int(d), int(f)))
