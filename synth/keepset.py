"""The 40-layer keep-set arena on the device: 40 layers x 154 resident experts of 384
(6,160 slots of 18,800,640 B, 115.8 GB) behind per-layer expert->slot tables whose kept
experts are drawn from a Zipf(1.1) popularity, plus each layer's router weight.  Input
generation only: the experts are the seeded synthetic tensors of synth.tensors, staged on the
device and packed by the library's own moe_pack_expert."""
from __future__ import annotations

import numpy as np

from . import gpu as sgpu
from . import tensors as syn

D, F, E, K, LAYERS, KEEP, ZIPF_S = 5120, 2304, 384, 6, 40, 154, 1.1
SCALE = (-10, -6)


def bits_to_device(bits: np.ndarray, device):
    """bf16 bit patterns (uint16) -> a torch bfloat16 tensor on `device`."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


class KeepSetArena:
    def __init__(self, device, seed: int = 0):
        import torch
        import fp4_routed_expert_gb300 as moe
        from fp4_routed_expert_gb300.layer import Arena
        self.seed = seed
        self.tabs = syn.keepset_slot_tables(seed, LAYERS, E, KEEP, ZIPF_S)
        self.dims = moe.moe_dims(D, F, E, K)
        self.arena = Arena(self.dims, LAYERS * KEEP, device)
        stage = sgpu.ExpertStaging(D, F, device)
        for l in range(LAYERS):
            for e in range(E):
                s = int(self.tabs[l, e])
                if s >= 0:
                    self.arena.pack(s, stage.fill(seed, l, e, *SCALE))
        torch.cuda.synchronize()
        del stage
        self.wr_bits = [syn.router_weight(seed, l, E, D) for l in range(LAYERS)]
        self.wr = [bits_to_device(b, device) for b in self.wr_bits]
        self.tab_dev = [torch.from_numpy(np.ascontiguousarray(self.tabs[l])).to(device) for l in range(LAYERS)]

    def release(self):
        del self.arena
