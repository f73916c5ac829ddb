"""The router entry point that allocates nothing (moe_route_topk_noalloc).

It serves callers that cannot allocate device memory -- an op hosted by an engine that owns
the whole device pool and gives its ops no workspace, or a serving loop that must not
allocate between steps -- by keeping its scratch in a static array inside the library.
These tests check, through the C ABI, that two calls in a row give the same ids, slots and
weights, bit for bit, as the workspace entry point moe_route_topk on the same inputs (both
run the same kernels), and the same ids and slots as the oracle.  The cases cover both
router paths it can take: the one-pass decode router (small d) and, when the tokens' rows do
not fit in shared memory (T = 16 at d = 6144), the norms -> tiled logits -> selection path on
the static array's slices.  This file is collected last so that a stop-at-first-failure run
has already run every other test."""
import ctypes

import numpy as np
import pytest

import fp4_routed_expert_gb300 as moe
import oracle
from synth import tensors as syn


def test_rejects_more_tokens_than_its_scratch_holds():
    L = moe.lib()
    dims = moe.moe_dims(512, 256, 16, 2)
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the size check answers first
    rc = L.moe_route_topk_noalloc(ctypes.byref(dims), 17, fake, fake, None, fake, fake, fake, fake, fake, None)
    assert rc == -3 and moe.moe_status_str(rc) == "token count out of range"


@pytest.mark.gpu
@pytest.mark.parametrize("d,E,T", [(1024, 96, 1), (1024, 96, 16), (6144, 40, 16)],
                         ids=["decode_router_T1", "decode_router_T16", "tiled_router_T16_d6144"])
def test_noalloc_router_matches_workspace_router_twice(d, E, T):
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    k = 6
    dims = moe.moe_dims(d, 256, E, k)
    to = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).to(dev).view(torch.bfloat16)
    wr = to(syn.router_weight(11, 0, E, d))
    table = syn.permuted_slot_table(11, 0, E)
    table[::5] = -1                                   # some experts without a slot
    tab = torch.from_numpy(table).to(dev)
    bias = torch.from_numpy(syn.zipf_score_bias(11, 0, E, 1.2, 0.04)).to(dev)
    ws = torch.empty(moe.moe_workspace_bytes(dims, T), dtype=torch.uint8, device=dev)
    moe.moe_workspace_init(dims, ws)

    def outputs():
        return (torch.empty((T, k), dtype=torch.int32, device=dev), torch.empty((T, k), dtype=torch.float32, device=dev),
                torch.empty((T, k), dtype=torch.int32, device=dev), torch.zeros(1, dtype=torch.int32, device=dev))

    wr_bits = syn.router_weight(11, 0, E, d)
    bias_np = syn.zipf_score_bias(11, 0, E, 1.2, 0.04)
    for call in range(2):
        x_bits = syn.activations(11, 0, T, d, stream=8 + call)
        x = to(x_bits)
        ids0, w0, s0, st0 = outputs()
        moe.moe_route_topk(dims, T, x, wr, bias, tab, ids0, w0, s0, st0, ws)
        ids1, w1, s1, st1 = outputs()
        moe.moe_route_topk_noalloc(dims, T, x, wr, bias, tab, ids1, w1, s1, st1)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(ids1.cpu().numpy(), ids0.cpu().numpy())
        np.testing.assert_array_equal(s1.cpu().numpy(), s0.cpu().numpy())
        np.testing.assert_array_equal(w1.cpu().numpy(), w0.cpu().numpy())
        assert int(st1.item()) == int(st0.item()) == 0
        ref = oracle.route_topk(x_bits, wr_bits, bias_np, table, k)
        np.testing.assert_array_equal(ids1.cpu().numpy(), ref["ids"])
        np.testing.assert_array_equal(s1.cpu().numpy(), ref["slots"])
        np.testing.assert_allclose(w1.cpu().numpy(), ref["weights"], rtol=2e-5, atol=1e-7)
