"""The cb3 slot layout as the kernel source documents it, written out on the host from random
levels and indices and read back by the decoder the GPU tests use (so that decoder is pinned
to the documented layout, not to the packer it checks)."""
import numpy as np

import fp4_routed_expert_gb300 as moe
from test_gpu_cb3 import cb3_decode_slot


def encode_slot(lv: dict, idx: dict, d: int, f: int) -> np.ndarray:
    """levels: 16 bytes per row (gate rows, up rows, down rows); then per row three word arrays
    A, B, Z of K/32 words; element j of group c with index v: (v & 3) in A at bit
    4(j%8) + 2(j/8) for j < 16, in B at bit 4(j%8) + 2((j-16)/8) for j >= 16, and (v >> 2) in Z
    at bit 4(j%8) + (2, 3, 0, 1)[j/8]."""
    R = 2 * f + d
    out = bytearray(moe.moe_cb3_slot_bytes((d, f, 16, 2)))
    levels = np.concatenate([lv["gate"], lv["up"], lv["down"]]).astype("<u2")
    out[:16 * R] = levels.tobytes()
    off = 16 * R
    for m, K in (("gate", d), ("up", d), ("down", f)):
        for row in idx[m]:
            nc = K // 32
            A = [0] * nc
            B = [0] * nc
            Z = [0] * nc
            for c in range(nc):
                for j in range(32):
                    v = int(row[32 * c + j])
                    if j < 16:
                        A[c] |= (v & 3) << (4 * (j % 8) + 2 * (j // 8))
                    else:
                        B[c] |= (v & 3) << (4 * (j % 8) + 2 * ((j - 16) // 8))
                    Z[c] |= (v >> 2) << (4 * (j % 8) + (2, 3, 0, 1)[j // 8])
            words = np.array(A + B + Z, dtype="<u4")
            out[off:off + words.nbytes] = words.tobytes()
            off += words.nbytes
    assert off <= len(out)
    return np.frombuffer(bytes(out), np.uint8)


def test_documented_layout_round_trip():
    rng = np.random.default_rng(9)
    d, f = 512, 256
    lv = {"gate": rng.integers(0, 65536, (f, 8)), "up": rng.integers(0, 65536, (f, 8)),
          "down": rng.integers(0, 65536, (d, 8))}
    idx = {"gate": rng.integers(0, 8, (f, d)), "up": rng.integers(0, 8, (f, d)), "down": rng.integers(0, 8, (d, f))}
    buf = encode_slot(lv, idx, d, f)
    got = cb3_decode_slot(buf, d, f)
    for m in ("gate", "up", "down"):
        np.testing.assert_array_equal(got[m + "_cb"], lv[m].astype(np.uint16))
        np.testing.assert_array_equal(got[m + "_idx"], idx[m].astype(np.uint8))
