"""Counter-based Philox4x32-10 generator (Salmon, Moraes, Dror, Shaw, "Parallel random
numbers: as easy as 1, 2, 3", SC'11), vectorised over numpy arrays.

Every synthetic tensor of the MoE workloads is a pure function of (seed, tag, element
index), so the CPU side (numpy, here) and the device side (``synth/csrc/synth_fill.cu``)
can regenerate any element independently.  This module holds no MoE arithmetic: it only
produces random 32-bit words and turns them into input tensors.

Stream definition used everywhere in this repository:
    key     = (seed, tag)                       two 32-bit words
    counter = (block, 0, 0, 0)                  block = 0, 1, 2, ...
    words   = philox4x32_10(counter, key)       four 32-bit words per block
    word i of a stream = output word (i % 4) of block (i // 4)
    byte i of a stream = byte (i % 4), little-endian, of word (i // 4)
"""
from __future__ import annotations

import numpy as np

_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85
_MASK = np.uint64(0xFFFFFFFF)
_S32 = np.uint64(32)


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Ten Philox4x32 rounds on counter arrays (uint64 arrays holding 32-bit values)."""
    c0 = np.asarray(c0, dtype=np.uint64)
    c1 = np.asarray(c1, dtype=np.uint64)
    c2 = np.asarray(c2, dtype=np.uint64)
    c3 = np.asarray(c3, dtype=np.uint64)
    ka, kb = int(k0) & 0xFFFFFFFF, int(k1) & 0xFFFFFFFF
    for _ in range(10):
        p0 = _M0 * c0
        p1 = _M1 * c2
        hi0, lo0 = p0 >> _S32, p0 & _MASK
        hi1, lo1 = p1 >> _S32, p1 & _MASK
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint64(ka)), lo1, (hi0 ^ c3 ^ np.uint64(kb)), lo0
        ka = (ka + _W0) & 0xFFFFFFFF
        kb = (kb + _W1) & 0xFFFFFFFF
    return c0, c1, c2, c3


def words(seed: int, tag: int, n: int, start: int = 0) -> np.ndarray:
    """Words [start, start+n) of the stream keyed by (seed, tag), as uint32."""
    if n <= 0:
        return np.zeros(0, dtype=np.uint32)
    b0 = start // 4
    b1 = (start + n + 3) // 4
    blocks = np.arange(b0, b1, dtype=np.uint64)
    if b1 > 0xFFFFFFFF:
        raise ValueError("stream longer than 2^32 blocks")
    z = np.zeros_like(blocks)
    o = philox4x32_10(blocks, z, z, z, seed, tag)
    w = np.stack(o, axis=1).reshape(-1).astype(np.uint32)
    off = start - 4 * b0
    return w[off:off + n]


def stream_bytes(seed: int, tag: int, n: int) -> np.ndarray:
    """Bytes [0, n) of the stream keyed by (seed, tag), as uint8."""
    w = words(seed, tag, (n + 3) // 4)
    return w.view(np.uint8)[:n].copy()


def uniform_ints(seed: int, tag: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers in [lo, hi]: word i of the stream taken modulo (hi-lo+1), plus lo."""
    span = hi - lo + 1
    w = words(seed, tag, n).astype(np.int64)
    return (lo + (w % span)).astype(np.int64)


def uniform01(seed: int, tag: int, n: int) -> np.ndarray:
    """n doubles strictly inside (0, 1): 53 bits from words (2i, 2i+1), plus half an ulp."""
    w = words(seed, tag, 2 * n).astype(np.uint64).reshape(n, 2)
    a = (w[:, 0] >> np.uint64(5)).astype(np.float64)
    b = (w[:, 1] >> np.uint64(6)).astype(np.float64)
    return (a * 67108864.0 + b + 0.5) / 9007199254740992.0


def normal(seed: int, tag: int, n: int) -> np.ndarray:
    """n standard normals (double) by Box-Muller on pairs of uniform01 draws."""
    m = (n + 1) // 2
    u = uniform01(seed, tag, 2 * m).reshape(m, 2)
    r = np.sqrt(-2.0 * np.log(u[:, 0]))
    th = 2.0 * np.pi * u[:, 1]
    z = np.stack([r * np.cos(th), r * np.sin(th)], axis=1).reshape(-1)
    return z[:n]
