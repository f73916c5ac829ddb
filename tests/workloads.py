"""Seeded workloads shared by the GPU tests: device arenas filled by the device generator
and packed through the library, plus the matching host tensors for the oracle."""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

import fp4_routed_expert_gb300 as moe
from fp4_routed_expert_gb300.layer import Arena, MoeLayer
from synth import gpu as sgpu
from synth import tensors as syn


def bits_to_torch(b: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).to(device).view(torch.bfloat16)


@dataclass
class Workload:
    d: int
    f: int
    E: int
    k: int
    seed: int
    layer: int
    scale_lo: int
    scale_hi: int
    table: np.ndarray            # expert -> slot
    wr: np.ndarray               # bf16 bits [E, d]
    bias: np.ndarray | None
    arena: Arena
    slot_expert: dict            # slot -> (layer, expert) whose tensors it holds

    def expert_tensors(self, slot: int) -> dict:
        layer, e = self.slot_expert[slot]
        return syn.expert_tensors(self.seed, layer, e, self.d, self.f, self.scale_lo, self.scale_hi)


def make_workload(d, f, E, k, seed=0, layer=0, scale=(-8, -4), table="identity", bias=None, num_slots=None,
                  device="cuda") -> Workload:
    if isinstance(table, str):
        table = syn.identity_slot_table(E) if table == "identity" else syn.permuted_slot_table(seed, layer, E)
    table = np.asarray(table, np.int32)
    dims = moe.moe_dims(d, f, E, k)
    ns = num_slots or int(max(table.max() + 1, 1))
    arena = Arena(dims, ns, device)
    stage = sgpu.ExpertStaging(d, f, device)
    slot_expert = {}
    for e in range(E):
        s = int(table[e])
        if s < 0:
            continue
        t = stage.fill(seed, layer, e, *scale)
        arena.pack(s, t)
        slot_expert[s] = (layer, e)
    torch.cuda.synchronize()
    wr = syn.router_weight(seed, layer, E, d)
    return Workload(d, f, E, k, seed, layer, scale[0], scale[1], table, wr, bias, arena, slot_expert)


def row_rel_err(y_gpu: np.ndarray, y_ref: np.ndarray) -> np.ndarray:
    """Per token row: max_i |y_gpu - y_ref| / max_i |y_ref|."""
    num = np.abs(y_gpu - y_ref).max(axis=1)
    den = np.abs(y_ref).max(axis=1)
    return num / np.maximum(den, 1e-30)


def elem_rel_err(y_gpu: np.ndarray, y_ref: np.ndarray, floor: float = 1e-3) -> np.ndarray:
    """Per token row: max_i |y_gpu - y_ref| / max(|y_ref_i|, floor * max_i |y_ref|), the
    elementwise relative error with a floor (reported beside the normwise row bound, which is
    the one asserted: a plain elementwise ratio is unbounded where y_ref is near 0)."""
    y_gpu = np.asarray(y_gpu, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    den = np.maximum(np.abs(y_ref), floor * np.abs(y_ref).max(axis=1, keepdims=True))
    return (np.abs(y_gpu - y_ref) / np.maximum(den, 1e-30)).max(axis=1)
