"""The C-ABI library loads and exports every entry point its header declares; host-side
argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

import fp4_routed_expert_gb300 as moe

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "fp4moe.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    L = moe.lib()
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n


def test_slot_bytes_and_workspace():
    assert moe.moe_slot_bytes((5120, 2304, 384, 6)) == 18_800_640
    assert moe.moe_slot_bytes((512, 256, 16, 2)) == 208_896
    assert moe.moe_slot_bytes((500, 256, 16, 2)) == -1
    assert moe.moe_slot_bytes((384, 256, 16, 2)) == -1      # d, f must be multiples of 256
    assert moe.moe_workspace_bytes((5120, 2304, 384, 6), 1) > 0
    assert moe.moe_workspace_bytes((5120, 2304, 384, 6), 4096) > moe.moe_workspace_bytes((5120, 2304, 384, 6), 16)
    assert moe.moe_workspace_bytes((5120, 2304, 2000, 6), 1) == 0
    # cb3: 16 bytes of levels per row (2f + d rows) + 3 bits per weight, rounded up to 1 KB
    assert moe.moe_cb3_slot_bytes((5120, 2304, 384, 6)) == 13_426_688
    assert moe.moe_cb3_slot_bytes((512, 256, 16, 2)) == 163_840
    assert moe.moe_cb3_slot_bytes((500, 256, 16, 2)) == -1


def test_host_argument_errors_return_before_any_launch():
    L = moe.lib()
    launched = moe.moe_kernel_launches()
    good = moe.moe_dims(512, 256, 16, 2)
    bad = moe.moe_dims(512, 256, 16, 40)
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: every call below fails its host checks first
    assert L.moe_route_topk(ctypes.byref(bad), 1, fake, fake, None, fake, fake, fake, fake, fake, fake, 1 << 30, None) == -2
    assert L.moe_route_topk(ctypes.byref(good), -1, fake, fake, None, fake, fake, fake, fake, fake, fake, 1 << 30, None) == -3
    assert L.moe_route_topk(ctypes.byref(good), 1, None, fake, None, fake, fake, fake, fake, fake, fake, 1 << 30, None) == -1
    assert L.moe_route_topk(ctypes.byref(good), 1, fake, fake, None, fake, fake, fake, fake, fake, fake, 16, None) == -4
    assert L.moe_route_topk(ctypes.byref(good), 1, P((1 << 20) + 2), fake, None, fake, fake, fake, fake, fake, fake, 1 << 30, None) == -8
    ar = moe.moe_arena(1 << 20, 12345, 4)
    assert L.moe_expert_ffn_fp4(ctypes.byref(good), ctypes.byref(ar), 1, fake, fake, fake, fake, None, None, None, 1,
                                None, fake, fake, fake, 1 << 30, None) == -5
    ar = moe.moe_arena(1 << 20, moe.moe_slot_bytes(good), 4)
    assert L.moe_expert_ffn_fp4(ctypes.byref(good), ctypes.byref(ar), 1, fake, fake, fake, fake, None, None, None, 7,
                                None, fake, fake, fake, 1 << 30, None) == -6
    assert L.moe_pack_expert(ctypes.byref(good), fake, fake, fake, fake, fake, fake, ctypes.byref(ar), 9, None) == -5
    assert L.moe_split_waves(ctypes.byref(good), 1, fake, fake, fake, 0, fake, fake, fake, fake, None) == -5
    assert L.moe_split_waves(ctypes.byref(good), 1, fake, None, fake, 4, fake, fake, fake, fake, None) == -1
    ar = moe.moe_arena(1 << 20, moe.moe_slot_bytes(good), 4)
    assert L.moe_gather_experts(ctypes.byref(good), ctypes.byref(ar), P((1 << 20) + 8), 16, fake, fake, fake, fake, fake,
                                None) == -8
    assert L.moe_gather_experts(ctypes.byref(good), ctypes.byref(ar), fake, 16, fake, None, fake, fake, fake, None) == -1
    f32 = ctypes.c_float
    assert L.moe_residency_bias(ctypes.byref(good), None, fake, fake, 0, f32(0.1), fake, None) == -5
    assert L.moe_residency_bias(ctypes.byref(good), None, fake, None, 4, f32(0.1), fake, None) == -1
    assert L.moe_residency_bias(ctypes.byref(good), None, fake, fake, 4, f32(-0.1), fake, None) == -2
    assert L.moe_residency_bias(ctypes.byref(good), None, fake, fake, 4, f32(float("nan")), fake, None) == -2
    assert L.moe_residency_bias(ctypes.byref(good), None, fake, fake, 4, f32(float("inf")), fake, None) == -2
    fp4_ar = moe.moe_arena(1 << 20, moe.moe_slot_bytes(good), 4)
    cb3_ar = moe.moe_arena(1 << 20, moe.moe_cb3_slot_bytes(good), 4)
    assert L.moe_pack_cb3(ctypes.byref(good), ctypes.byref(fp4_ar), 0, ctypes.byref(fp4_ar), 0, fake, None) == -5
    assert L.moe_pack_cb3(ctypes.byref(good), ctypes.byref(fp4_ar), 4, ctypes.byref(cb3_ar), 0, fake, None) == -5
    assert L.moe_pack_cb3(ctypes.byref(good), ctypes.byref(fp4_ar), 0, ctypes.byref(cb3_ar), -1, fake, None) == -5
    assert L.moe_pack_cb3(ctypes.byref(good), ctypes.byref(fp4_ar), 0, ctypes.byref(cb3_ar), 0, None, None) == -1
    assert L.moe_pack_cb3(ctypes.byref(bad), ctypes.byref(fp4_ar), 0, ctypes.byref(cb3_ar), 0, fake, None) == -2
    assert L.moe_expert_ffn_cb3(ctypes.byref(good), ctypes.byref(cb3_ar), -1, fake, fake, fake, fake, fake, fake,
                                1 << 30, None) == -3
    assert L.moe_expert_ffn_cb3(ctypes.byref(good), ctypes.byref(fp4_ar), 1, fake, fake, fake, fake, fake, fake,
                                1 << 30, None) == -5
    assert L.moe_expert_ffn_cb3(ctypes.byref(good), ctypes.byref(cb3_ar), 1, fake, fake, fake, None, fake, fake,
                                1 << 30, None) == -1
    assert L.moe_expert_ffn_cb3(ctypes.byref(good), ctypes.byref(cb3_ar), 1, fake, fake, fake, fake, fake, fake,
                                16, None) == -4
    lay = L.moe_layer_decode_fp4
    ok_ar = moe.moe_arena(1 << 20, moe.moe_slot_bytes(good), 4)
    bad_ar = moe.moe_arena(1 << 20, 12345, 4)
    args = lambda d, ar, T, x=fake, y=fake, wsb=1 << 30: (ctypes.byref(d), ctypes.byref(ar), T, x, fake, None, fake,
                                                        fake, fake, fake, y, fake, fake, wsb, None)
    assert lay(*args(bad, ok_ar, 1)) == -2
    assert lay(*args(good, ok_ar, 17)) == -3                  # decode only: T <= 16
    assert lay(*args(good, ok_ar, -1)) == -3
    assert lay(*args(good, bad_ar, 1)) == -5
    assert lay(*args(good, ok_ar, 1, y=None)) == -1
    assert lay(*args(good, ok_ar, 1, x=P((1 << 20) + 2))) == -8
    assert lay(*args(good, ok_ar, 1, wsb=16)) == -4
    cr = L.moe_expert_ffn_cb3_rows
    assert cr(ctypes.byref(good), ctypes.byref(cb3_ar), -1, fake, fake, fake, fake, fake, fake, 1 << 30, None) == -3
    assert cr(ctypes.byref(good), ctypes.byref(fp4_ar), 1, fake, fake, fake, fake, fake, fake, 1 << 30, None) == -5
    assert cr(ctypes.byref(good), ctypes.byref(cb3_ar), 1, fake, fake, fake, None, fake, fake, 1 << 30, None) == -1
    assert cr(ctypes.byref(good), ctypes.byref(cb3_ar), 1, fake, fake, fake, fake, fake, fake, 16, None) == -4
    assert moe.moe_status_str(-4) == "workspace too small"
    assert moe.moe_kernel_launches() == launched      # every rejected call launched nothing
