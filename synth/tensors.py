"""Seeded synthetic inputs for the routed-expert MoE layer (CPU side, numpy).

Nothing here computes the layer: it draws codes, scale bytes, activations, router weights,
score biases, expert->slot tables and keep-sets.  Integer tensors (the FP4 codes and UE8M0
scale bytes that fill the expert arena) are a pure function of (seed, tag, index) through
the Philox stream in ``synth.philox``, and ``synth/csrc/synth_fill.cu`` produces the same
bytes on the device.  Floating-point inputs are drawn on the CPU only.

Canonical (checkpoint-like) expert layout, K-contiguous, two codes per byte with element
2i in the low nibble:
    gate_q, up_q : uint8 [f, d/2]     gate_s, up_s : uint8 [f, d/32]
    down_q       : uint8 [d, f/2]     down_s       : uint8 [d, f/32]
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import philox

# Tensor kinds, placed in the top 4 bits of the 32-bit tag.
KIND_GATE_Q, KIND_GATE_S, KIND_UP_Q, KIND_UP_S, KIND_DOWN_Q, KIND_DOWN_S = range(6)
KIND_X = 8
KIND_ROUTER = 9
KIND_BIAS_PERM = 10
KIND_SLOT_PERM = 11
KIND_KEEP = 12
KIND_KEEP_SLOTS = 13

EXPERT_TENSORS = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")


def tag(kind: int, layer: int = 0, index: int = 0) -> int:
    """32-bit stream tag: kind (4 bits) | layer (8 bits) | index (20 bits)."""
    if not (0 <= kind < 16 and 0 <= layer < 256 and 0 <= index < (1 << 20)):
        raise ValueError("tag field out of range")
    return (kind << 28) | (layer << 20) | index


def expert_tensor_shapes(d: int, f: int) -> dict:
    return {
        "gate_q": (f, d // 2), "gate_s": (f, d // 32),
        "up_q": (f, d // 2), "up_s": (f, d // 32),
        "down_q": (d, f // 2), "down_s": (d, f // 32),
    }


def expert_tensors(seed: int, layer: int, expert: int, d: int, f: int,
                   scale_lo: int, scale_hi: int) -> dict:
    """The six canonical tensors of one expert.

    Codes are uniform bytes (so every nibble is uniform over all 16 e2m1 codes).
    Scale bytes are 127 + U{scale_lo..scale_hi}: word i of the stream modulo the span.
    """
    shapes = expert_tensor_shapes(d, f)
    out = {}
    for kind, name in enumerate(EXPERT_TENSORS):
        shp = shapes[name]
        n = shp[0] * shp[1]
        t = tag(kind, layer, expert)
        if name.endswith("_q"):
            out[name] = philox.stream_bytes(seed, t, n).reshape(shp)
        else:
            out[name] = (127 + philox.uniform_ints(seed, t, n, scale_lo, scale_hi)
                         ).astype(np.uint8).reshape(shp)
    return out


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def activations(seed: int, layer: int, T: int, d: int, start_token: int = 0,
                stream: int = 0) -> np.ndarray:
    """x [T, d] as bf16 bits: N(0,1) drawn in double, rounded to fp32, then to bf16.

    Token t of the stream uses words from row (start_token + t), so any subset of tokens
    can be regenerated alone.  ``stream`` (0..15) selects independent token streams of up
    to 65,536 tokens each.
    """
    if not (0 <= stream < 16 and 0 <= start_token and start_token + T <= 65536):
        raise ValueError("activation stream must be 0..15 with at most 65,536 tokens")
    rows = []
    for t in range(start_token, start_token + T):
        z = philox.normal(seed, tag(KIND_X, layer, (stream << 16) + t) , d)
        rows.append(f32_to_bf16_bits(z.astype(np.float32)))
    return np.stack(rows) if rows else np.zeros((0, d), np.uint16)


def router_weight(seed: int, layer: int, E: int, d: int, std: float = 0.02) -> np.ndarray:
    """W_r [E, d] as bf16 bits, N(0, std^2)."""
    z = philox.normal(seed, tag(KIND_ROUTER, layer, 0), E * d) * std
    return f32_to_bf16_bits(z.astype(np.float32)).reshape(E, d)


def seeded_permutation(seed: int, t: int, n: int) -> np.ndarray:
    """A permutation of range(n): stable argsort of n 32-bit stream words."""
    w = philox.words(seed, t, n).astype(np.int64)
    return np.argsort(w, kind="stable").astype(np.int64)


def zipf_score_bias(seed: int, layer: int, E: int, s: float, beta: float) -> np.ndarray:
    """Per-expert score bias b_e = beta * (ln p_e - mean_e ln p_e), p_e ~ (rank_e + 1)^-s.

    rank_e comes from a seeded permutation, so popularity is spread over expert ids.
    Returned as float32 [E].
    """
    rank = np.empty(E, np.int64)
    rank[seeded_permutation(seed, tag(KIND_BIAS_PERM, layer, 0), E)] = np.arange(E)
    lp = -s * np.log(rank + 1.0)
    return (beta * (lp - lp.mean())).astype(np.float32)


def permuted_slot_table(seed: int, layer: int, E: int) -> np.ndarray:
    """expert -> slot, a random permutation of 0..E-1 (int32)."""
    return seeded_permutation(seed, tag(KIND_SLOT_PERM, layer, 0), E).astype(np.int32)


def identity_slot_table(E: int) -> np.ndarray:
    return np.arange(E, dtype=np.int32)


def keep_set(seed: int, layer: int, E: int, keep: int, s: float) -> np.ndarray:
    """Sorted expert ids kept resident in one layer: `keep` draws without replacement from
    a Zipf(s) popularity over a seeded ranking (Efraimidis-Spirakis keys u^(1/p))."""
    rank = np.empty(E, np.int64)
    rank[seeded_permutation(seed, tag(KIND_KEEP, layer, 0), E)] = np.arange(E)
    p = (rank + 1.0) ** (-s)
    p /= p.sum()
    u = philox.uniform01(seed, tag(KIND_KEEP, layer, 1), E)
    keys = np.log(u) / p          # monotone in u^(1/p)
    chosen = np.argsort(-keys, kind="stable")[:keep]
    return np.sort(chosen)


def keepset_slot_tables(seed: int, layers: int, E: int, keep: int, s: float) -> np.ndarray:
    """[layers, E] expert->slot tables over one shared arena of layers*keep slots.

    Non-resident experts map to -1.  Slot numbers are a seeded permutation of
    0..layers*keep-1 assigned to (layer, kept expert) pairs in order.
    """
    n = layers * keep
    perm = seeded_permutation(seed, tag(KIND_KEEP_SLOTS, 0, 0), n)
    tab = np.full((layers, E), -1, np.int32)
    i = 0
    for l in range(layers):
        for e in keep_set(seed, l, E, keep, s):
            tab[l, e] = perm[i]
            i += 1
    return tab


@dataclass(frozen=True)
class LayerShape:
    d: int
    f: int
    E: int
    k: int

    @property
    def expert_bytes(self) -> int:
        # three [f x d] matrices: half a byte per code plus one scale byte per 32 codes
        return 3 * self.f * self.d // 2 + 3 * self.f * self.d // 32
