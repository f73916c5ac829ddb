"""One routed-expert MoE layer on the device: owns the buffers and issues the C-ABI calls in
order on one stream.  This is argument marshalling only; the arithmetic is in the library."""
from __future__ import annotations

import torch

from . import (DECODE_MAX_T, MOE_FFN_CUDA_CORES, MOE_FUSE_COMBINE, moe_arena, moe_cb3_slot_bytes, moe_dims,
               moe_expert_ffn_cb3, moe_expert_ffn_fp4, moe_layer_decode_fp4, moe_pack_cb3, moe_pack_expert,
               moe_permute, moe_route_topk, moe_slot_bytes, moe_workspace_bytes, moe_workspace_init)


def aligned_empty(nbytes: int, align: int = 1024, device=None) -> torch.Tensor:
    """A uint8 CUDA buffer of nbytes whose start is aligned to `align` bytes."""
    raw = torch.empty(nbytes + align, dtype=torch.uint8, device=device)
    off = (-raw.data_ptr()) % align
    return raw[off:off + nbytes]


class Arena:
    """Resident expert slots (device memory)."""

    def __init__(self, dims: moe_dims, num_slots: int, device=None):
        self.dims = dims
        self.slot_bytes = moe_slot_bytes(dims)
        if self.slot_bytes <= 0:
            raise ValueError("unsupported dims")
        self.buf = aligned_empty(self.slot_bytes * num_slots, 1024, device)
        self.c = moe_arena(self.buf.data_ptr(), self.slot_bytes, num_slots)
        self.num_slots = num_slots

    def pack(self, slot: int, t: dict, stream=None):
        moe_pack_expert(self.dims, t["gate_q"], t["gate_s"], t["up_q"], t["up_s"], t["down_q"], t["down_s"],
                        self.c, slot, stream)


class Cb3Arena:
    """Resident expert slots in the cb3 format (3-bit per-row codebook), packed on the device
    from FP4 slots."""

    def __init__(self, dims: moe_dims, num_slots: int, device=None):
        self.dims = dims
        self.slot_bytes = moe_cb3_slot_bytes(dims)
        if self.slot_bytes <= 0:
            raise ValueError("unsupported dims")
        self.buf = aligned_empty(self.slot_bytes * num_slots, 1024, device)
        self.c = moe_arena(self.buf.data_ptr(), self.slot_bytes, num_slots)
        self.num_slots = num_slots

    def pack_from(self, fp4: Arena, fp4_slot: int, slot: int, status, stream=None):
        moe_pack_cb3(self.dims, fp4.c, fp4_slot, self.c, slot, status, stream)


class MoeLayer:
    """Buffers for up to T_max tokens and the call sequence of one layer.

    Decode (T <= 16): route -> experts with the combine fused.
    Prefill: route -> permute -> experts (rows) -> combine, or experts with the combine fused.
    """

    def __init__(self, d: int, f: int, E: int, k: int, T_max: int, arena: Arena, device=None):
        self.dims = moe_dims(d, f, E, k)
        self.arena = arena
        self.T_max = T_max
        dev = device or torch.device("cuda", torch.cuda.current_device())
        self.ws = aligned_empty(moe_workspace_bytes(self.dims, T_max), 256, dev)
        moe_workspace_init(self.dims, self.ws)
        n = max(T_max, 1) * k
        self.ids = torch.empty((max(T_max, 1), k), dtype=torch.int32, device=dev)
        self.w = torch.empty((max(T_max, 1), k), dtype=torch.float32, device=dev)
        self.slots = torch.empty((max(T_max, 1), k), dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        self.row_src = torch.empty(n, dtype=torch.int32, device=dev)
        self.row_dst = torch.empty(n, dtype=torch.int32, device=dev)
        self.rows = torch.empty((n, d), dtype=torch.float32, device=dev) if T_max > DECODE_MAX_T else None
        self.y = torch.empty((max(T_max, 1), d), dtype=torch.bfloat16, device=dev)

    def experts_cb3(self, cb3: Cb3Arena, x, T=None, stream=None, y=None):
        """Expert FFN + combine on cb3 experts (any T: more than 16 tokens as consecutive calls
        of 16); the routing's slots index the cb3 arena."""
        T = x.shape[0] if T is None else T
        y = self.y if y is None else y
        moe_expert_ffn_cb3(self.dims, cb3.c, T, x, self.slots, self.w, y, self.status, self.ws, stream)
        return y

    def route(self, x, w_router, table, bias=None, T=None, stream=None):
        T = x.shape[0] if T is None else T
        moe_route_topk(self.dims, T, x, w_router, bias, table, self.ids, self.w, self.slots, self.status, self.ws,
                       stream)

    def experts(self, x, T=None, fused_prefill=False, stream=None, y=None, cuda_cores=False):
        """Expert FFN + combine.  cuda_cores=True selects the CUDA-core kernels (exact fp4 x bf16
        products: the streaming kernel in decode, grouped GEMMs in prefill); the default uses the
        tensor-core kernels where the shape allows."""
        T = x.shape[0] if T is None else T
        y = self.y if y is None else y
        extra = MOE_FFN_CUDA_CORES if cuda_cores else 0
        if T <= DECODE_MAX_T:
            moe_expert_ffn_fp4(self.dims, self.arena.c, T, x, self.ids, self.slots, self.w, None, None, None,
                               MOE_FUSE_COMBINE | extra, None, y, self.status, self.ws, stream)
            return y
        moe_permute(self.dims, T, self.ids, self.offsets, self.row_src, self.row_dst, self.ws, stream)
        if fused_prefill:
            moe_expert_ffn_fp4(self.dims, self.arena.c, T, x, self.ids, self.slots, self.w, self.offsets,
                               self.row_src, self.row_dst, MOE_FUSE_COMBINE | extra, None, y, self.status, self.ws,
                               stream)
        else:
            from . import moe_combine
            moe_expert_ffn_fp4(self.dims, self.arena.c, T, x, self.ids, self.slots, self.w, self.offsets,
                               self.row_src, self.row_dst, extra, self.rows, None, self.status, self.ws, stream)
            moe_combine(self.dims, T, self.rows, self.row_dst, self.w, y, stream)
        return y

    def decode(self, x, w_router, table, bias=None, T=None, stream=None, y=None):
        """Routing, expert FFN and combine of a decode call (T <= 16) in one request
        (moe_layer_decode_fp4): the same outputs as route() then experts()."""
        T = x.shape[0] if T is None else T
        y = self.y if y is None else y
        moe_layer_decode_fp4(self.dims, self.arena.c, T, x, w_router, bias, table, self.ids, self.w, self.slots, y,
                             self.status, self.ws, stream)
        return y

    def forward(self, x, w_router, table, bias=None, stream=None, y=None, cuda_cores=False):
        self.route(x, w_router, table, bias, stream=stream)
        return self.experts(x, stream=stream, y=y, cuda_cores=cuda_cores)
