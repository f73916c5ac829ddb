"""Device-side synthetic expert tensors (same bytes as synth.tensors.expert_tensors)."""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import tensors as syn

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc", "synth_fill.cu")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    os.makedirs(OUT, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    nvcc = "/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else "nvcc"
    tmp = LIB + ".tmp.%d" % os.getpid()
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-Xcompiler", "-fPIC",
                           "-shared", "-cudart", "shared", "-o", tmp, SRC])
    os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        L.synth_fill_bytes.restype = ctypes.c_int
        L.synth_fill_bytes.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_void_p]
        L.synth_fill_scales.restype = ctypes.c_int
        L.synth_fill_scales.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_uint32, ctypes.c_uint32,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
        _lib = L
    return _lib


class ExpertStaging:
    """Device buffers for one expert's canonical tensors, refilled per expert."""

    def __init__(self, d: int, f: int, device):
        import torch
        self.shapes = syn.expert_tensor_shapes(d, f)
        self.t = {n: torch.empty(s, dtype=torch.uint8, device=device) for n, s in self.shapes.items()}

    def fill(self, seed: int, layer: int, expert: int, scale_lo: int, scale_hi: int, stream=None):
        import torch
        st = ctypes.c_void_p((torch.cuda.current_stream() if stream is None else stream).cuda_stream)
        L = lib()
        for kind, name in enumerate(syn.EXPERT_TENSORS):
            buf = self.t[name]
            tg = syn.tag(kind, layer, expert)
            if name.endswith("_q"):
                rc = L.synth_fill_bytes(ctypes.c_void_p(buf.data_ptr()), buf.numel(), seed, tg, st)
            else:
                rc = L.synth_fill_scales(ctypes.c_void_p(buf.data_ptr()), buf.numel(), seed, tg, scale_lo, scale_hi, st)
            if rc != 0:
                raise RuntimeError("synth fill failed: %d" % rc)
        return self.t
