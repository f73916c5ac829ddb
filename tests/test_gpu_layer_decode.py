"""moe_layer_decode_fp4: routing and experts of a decode call in one request.  On the tensor-core
path with at most 384 experts the router kernel only writes its key records and the expert
kernel selects from them itself; the outputs must equal those of moe_route_topk followed by
moe_expert_ffn_fp4 bit for bit, and match the oracle."""
import numpy as np
import pytest
import torch

import fp4_routed_expert_gb300 as moe
from fp4_routed_expert_gb300.layer import MoeLayer
from synth import tensors as syn

from test_gpu_parity import check_tokens, run_layer
from workloads import bits_to_torch, make_workload

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_fused(wl, x_bits, bias=None, table=None, layer=None):
    T = x_bits.shape[0]
    layer = layer or MoeLayer(wl.d, wl.f, wl.E, wl.k, max(T, 1), wl.arena)
    x = bits_to_torch(x_bits, DEV)
    wr = bits_to_torch(wl.wr, DEV)
    tab = torch.from_numpy(wl.table if table is None else table).to(DEV)
    b = None if bias is None else torch.from_numpy(bias).to(DEV)
    y = layer.decode(x, wr, tab, b)
    torch.cuda.synchronize()
    return dict(ids=layer.ids[:T].cpu().numpy(), w=layer.w[:T].cpu().numpy(), slots=layer.slots[:T].cpu().numpy(),
                status=int(layer.status.item()), y=y[:T].float().cpu().numpy())


def assert_same(a, b):
    assert a["status"] == b["status"]
    for key in ("ids", "slots", "w", "y"):
        assert a[key].tobytes() == b[key].tobytes(), key


@pytest.mark.parametrize("T", [1, 3, 8, 9, 16])
def test_fused_equals_separate_calls_ties_bias_mask(T):
    """40 experts (the expert kernel's 4-per-lane selection), exact ties between experts 3, 7
    and 21, a score bias, and a keep-set mask."""
    d, E, k = 512, 40, 4
    wl = make_workload(d, 256, E, k, seed=5, scale=(-8, -4))
    wr = wl.wr.copy()
    wr[7] = wr[3]
    wr[21] = wr[3]
    wl.wr = wr
    x = syn.activations(5, 0, T, d)
    fused = run_fused(wl, x)
    assert_same(fused, run_layer(wl, x))
    check_tokens(wl, x, fused, list(range(T)))
    bias = syn.zipf_score_bias(5, 0, E, 1.2, 0.5)
    fused = run_fused(wl, x, bias=bias)
    assert_same(fused, run_layer(wl, x, bias=bias))
    check_tokens(wl, x, fused, list(range(T)), bias=bias)
    tab = wl.table.copy()
    tab[::2] = -1
    wl.table = tab
    fused = run_fused(wl, x)
    assert np.all(fused["ids"] % 2 == 1)
    assert_same(fused, run_layer(wl, x))


def test_fused_few_resident_and_bad_slot():
    d, E, k = 512, 16, 4
    wl = make_workload(d, 256, E, k, seed=6, num_slots=16)
    x = syn.activations(6, 0, 2, d)
    tab = np.full(E, -1, np.int32)
    tab[[5, 9]] = [5, 9]
    wl.table = tab
    fused = run_fused(wl, x)
    assert fused["status"] & moe.MOE_STATUS_FEW_RESIDENT
    assert fused["ids"].tolist() == [[5, 9, -1, -1]] * 2
    assert_same(fused, run_layer(wl, x))
    tab = np.full(E, 100, np.int32)   # every slot outside the arena
    wl.table = tab
    fused = run_fused(wl, x)
    assert fused["status"] & moe.MOE_STATUS_BAD_SLOT
    assert np.all(fused["y"] == 0)


def test_fused_and_separate_calls_interleaved_on_one_workspace():
    """The hand-over counter is the separate router's ticket too: fused, separate and fused
    calls back to back on one workspace and one stream, without a synchronisation between
    them, each equal to its own separate-call reference."""
    d, E, k, T = 512, 64, 4, 2
    wl = make_workload(d, 256, E, k, seed=8, table="permuted", scale=(-8, -4))
    xs = [syn.activations(8, 0, T, d, stream=s) for s in range(6)]
    refs = [run_layer(wl, x) for x in xs]
    layer = MoeLayer(d, 256, E, k, T, wl.arena)
    wr = bits_to_torch(wl.wr, DEV)
    tab = torch.from_numpy(wl.table).to(DEV)
    ys = [torch.empty((T, d), dtype=torch.bfloat16, device=DEV) for _ in xs]
    ids = []
    for i, x in enumerate(xs):
        xt = bits_to_torch(x, DEV)
        if i % 3 == 1:
            layer.route(xt, wr, tab)
            layer.experts(xt, y=ys[i])
        else:
            layer.decode(xt, wr, tab, y=ys[i])
        ids.append(layer.ids[:T].clone())
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    for i, r in enumerate(refs):
        assert ids[i].cpu().numpy().tobytes() == r["ids"].tobytes(), i
        assert ys[i].float().cpu().numpy().tobytes() == r["y"].tobytes(), i


def test_fused_graph_replays_equal_eager():
    """A CUDA graph of 8 fused calls (the bench's form), replayed twice: every output equals
    the eager separate calls."""
    d, E, k, T, N = 512, 64, 4, 1, 8
    wl = make_workload(d, 256, E, k, seed=9, table="permuted", scale=(-8, -4))
    x = syn.activations(9, 0, N * T, d)
    layer = MoeLayer(d, 256, E, k, T, wl.arena)
    xt = bits_to_torch(x, DEV)
    wr = bits_to_torch(wl.wr, DEV)
    tab = torch.from_numpy(wl.table).to(DEV)
    y = torch.empty((N * T, d), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        layer.decode(xt[:T], wr, tab, y=y[:T])   # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(N):
            layer.decode(xt[i * T:(i + 1) * T], wr, tab, y=y[i * T:(i + 1) * T])
    for _ in range(2):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(layer.status.item()) == 0
        for i in range(N):
            ref = run_layer(wl, x[i * T:(i + 1) * T])
            assert y[i * T:(i + 1) * T].float().cpu().numpy().tobytes() == ref["y"].tobytes(), i


def test_fused_more_than_384_experts_takes_separate_launches():
    d, E, k, T = 256, 400, 6, 3
    wl = make_workload(d, 256, E, k, seed=10, table="permuted", scale=(-8, -4))
    x = syn.activations(10, 0, T, d)
    before = moe.moe_kernel_launches()
    fused = run_fused(wl, x)
    assert moe.moe_kernel_launches() - before == 2
    assert_same(fused, run_layer(wl, x))


@pytest.fixture(scope="module")
def full_decode():
    """d=5120, f=2304, E=384, k=6 (the expert kernel's 12-per-lane selection)."""
    return make_workload(5120, 2304, 384, 6, seed=0, table="permuted", scale=(-10, -6))


def test_fused_full_shape_decode_and_verify(full_decode):
    wl = full_decode
    x = syn.activations(0, 0, 16, 5120, stream=12)
    for t in range(2):
        fused = run_fused(wl, x[t:t + 1])
        assert_same(fused, run_layer(wl, x[t:t + 1]))
        check_tokens(wl, x[t:t + 1], fused, [0])
    fused = run_fused(wl, x)
    assert_same(fused, run_layer(wl, x))
    check_tokens(wl, x, fused, [0, 15])
