"""GPU parity: the CUDA library, called through its C ABI, against the CPU oracle on the same
seeded inputs.  Routing ids, slots and the permutation must match bit for bit; layer outputs
must satisfy the per-row bound max|y_gpu - y_ref| / max|y_ref| <= 1e-2."""
import numpy as np
import pytest
import torch

import fp4_routed_expert_gb300 as moe
from fp4_routed_expert_gb300.layer import Arena, MoeLayer
import oracle
from synth import gpu as sgpu
from synth import tensors as syn

from workloads import bits_to_torch, elem_rel_err, make_workload, row_rel_err

pytestmark = pytest.mark.gpu
TOL = 1e-2
DEV = "cuda"


def run_layer(wl, x_bits, bias=None, fused_prefill=False, cuda_cores=False):
    """cuda_cores=False: the tensor-core kernels (the default); True: the CUDA-core kernels
    (decode: the streaming kernel and its combine; prefill: grouped GEMMs)."""
    T = x_bits.shape[0]
    layer = MoeLayer(wl.d, wl.f, wl.E, wl.k, max(T, 1), wl.arena)
    x = bits_to_torch(x_bits, DEV)
    wr = bits_to_torch(wl.wr, DEV)
    tab = torch.from_numpy(wl.table).to(DEV)
    b = None if bias is None else torch.from_numpy(bias).to(DEV)
    layer.route(x, wr, tab, b)
    y = layer.experts(x, fused_prefill=fused_prefill, cuda_cores=cuda_cores)
    torch.cuda.synchronize()
    out = dict(ids=layer.ids[:T].cpu().numpy(), w=layer.w[:T].cpu().numpy(), slots=layer.slots[:T].cpu().numpy(),
               status=int(layer.status.item()), y=y[:T].float().cpu().numpy())
    if T > moe.DECODE_MAX_T:
        n = T * wl.k
        out["offsets"] = layer.offsets.cpu().numpy()
        out["row_src"] = layer.row_src[:n].cpu().numpy()
        out["row_dst"] = layer.row_dst[:n].cpu().numpy()
    return out


def oracle_tokens(wl, x_bits, tokens, bias=None):
    """Oracle routing and output for the given token indices (one by one)."""
    r = oracle.route_topk(x_bits[tokens], wl.wr, bias, wl.table, wl.k)
    ys = []
    cache = {}
    for n, t in enumerate(tokens):
        z = np.zeros((wl.k, wl.d), np.float32)
        for j in range(wl.k):
            s = int(r["slots"][n, j])
            if s < 0:
                continue
            if s not in cache:
                cache[s] = wl.expert_tensors(s)
            _, z[j] = oracle.expert_ffn_f32(x_bits[t], cache[s])
        ys.append(oracle.combine_f32(z, r["weights"][n]))
    return r, np.stack(ys)


def check_tokens(wl, x_bits, got, tokens, bias=None):
    r, y = oracle_tokens(wl, x_bits, tokens, bias)
    np.testing.assert_array_equal(got["ids"][tokens], r["ids"])
    np.testing.assert_array_equal(got["slots"][tokens], r["slots"])
    np.testing.assert_allclose(got["w"][tokens], r["weights"], rtol=2e-5, atol=1e-7)
    err = row_rel_err(got["y"][tokens], y)
    eerr = elem_rel_err(got["y"][tokens], y)
    print("max row error %.3e, elementwise (1e-3 floor) %.3e over %d tokens" % (err.max(), eerr.max(), len(tokens)))
    assert err.max() <= TOL, err
    return r


# ---------------------------------------------------------------------------- generator

def test_device_generator_matches_host():
    st = sgpu.ExpertStaging(512, 256, DEV)
    t = st.fill(0, 3, 11, -10, -6)
    torch.cuda.synchronize()
    ref = syn.expert_tensors(0, 3, 11, 512, 256, -10, -6)
    for n in syn.EXPERT_TENSORS:
        np.testing.assert_array_equal(t[n].cpu().numpy(), ref[n])


# ---------------------------------------------------------------------------- tiny workload

@pytest.fixture(scope="module")
def tiny():
    return make_workload(512, 256, 16, 2, seed=0, scale=(-8, -4))


def test_tiny_layer_matches_oracle(tiny):
    x = syn.activations(0, 0, 4, 512)
    got = run_layer(tiny, x)
    assert got["status"] == 0
    slots = {n: np.stack([tiny.expert_tensors(s)[n] for s in range(16)]) for n in syn.EXPERT_TENSORS}
    ref = oracle.moe_layer(x, tiny.wr, None, tiny.table, 2, slots)
    np.testing.assert_array_equal(got["ids"], ref["ids"])
    np.testing.assert_array_equal(got["slots"], ref["slots"])
    np.testing.assert_allclose(got["w"], ref["weights"], rtol=2e-5)
    assert row_rel_err(got["y"], ref["y"]).max() <= TOL


def oracle_with_routing(wl, x_bits, r):
    """Oracle layer output for tokens x_bits under the given routing (ids, slots, weights)."""
    cache, ys = {}, []
    for t in range(x_bits.shape[0]):
        z = np.zeros((wl.k, wl.d), np.float32)
        for j in range(wl.k):
            s = int(r["slots"][t, j])
            if s < 0:
                continue
            if s not in cache:
                cache[s] = wl.expert_tensors(s)
            _, z[j] = oracle.expert_ffn_f32(x_bits[t], cache[s])
        ys.append(oracle.combine_f32(z, r["weights"][t]))
    return np.stack(ys)


def test_back_to_back_calls_share_one_workspace(tiny):
    """Router and expert calls enqueued back to back on one stream and one workspace with no
    host synchronisation: a launch may start while the one before it still runs, and must
    neither disturb it nor see its state.  FFN after FFN (other activations, same routing),
    router after FFN and FFN after router, each output against the oracle."""
    T = 3
    xs = [syn.activations(0, 40 + i, T, 512) for i in range(2)]
    layer = MoeLayer(tiny.d, tiny.f, tiny.E, tiny.k, T, tiny.arena)
    xt = [bits_to_torch(x, DEV) for x in xs]
    wr = bits_to_torch(tiny.wr, DEV)
    tab = torch.from_numpy(tiny.table).to(DEV)
    outs = []
    layer.route(xt[0], wr, tab)
    for rep in range(4):                      # four FFN calls in a row on the first routing
        outs.append((0, rep % 2, layer.experts(xt[rep % 2], y=torch.empty((T, tiny.d), dtype=torch.bfloat16, device=DEV))))
    layer.route(xt[1], wr, tab)
    outs.append((1, 1, layer.experts(xt[1], y=torch.empty((T, tiny.d), dtype=torch.bfloat16, device=DEV))))
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    routes = [oracle.route_topk(x, tiny.wr, None, tiny.table, tiny.k) for x in xs]
    np.testing.assert_array_equal(layer.ids[:T].cpu().numpy(), routes[1]["ids"])
    for ri, xi, y in outs:
        ref = oracle_with_routing(tiny, xs[xi], routes[ri])
        err = row_rel_err(y.float().cpu().numpy(), ref)
        assert err.max() <= TOL, (ri, xi, err)


@pytest.mark.parametrize("cuda_cores", [False, True], ids=["tensor_cores", "cuda_cores"])
@pytest.mark.parametrize("T", [1, 3, 16, 17, 100])
def test_tiny_shapes_decode_and_prefill(tiny, T, cuda_cores):
    x = syn.activations(0, 0, T, 512, stream=1)
    got = run_layer(tiny, x, cuda_cores=cuda_cores)
    r = check_tokens(tiny, x, got, list(range(T)))
    if T > moe.DECODE_MAX_T:
        p = oracle.permute(r["ids"], 16)
        np.testing.assert_array_equal(got["offsets"], p["offsets"])
        np.testing.assert_array_equal(got["row_src"][:p["rows"]], p["row_src"])
        np.testing.assert_array_equal(got["row_dst"], p["row_dst"])


@pytest.fixture(scope="module")
def small_multistage():
    # d = 1024, f = 768: gate/up units of 4 K blocks (two pipeline stages), down units of 3 K
    # blocks (a full and a half stage, cut into two parts by the decode schedule)
    return make_workload(1024, 768, 16, 4, seed=5, scale=(-9, -5))


@pytest.mark.parametrize("T", [1, 2, 5, 17, 40])
def test_small_multistage_shape(small_multistage, T):
    x = syn.activations(5, 0, T, 1024)
    got = run_layer(small_multistage, x)
    assert got["status"] == 0
    check_tokens(small_multistage, x, got, list(range(T)))


@pytest.mark.parametrize("cuda_cores", [False, True], ids=["tensor_cores", "cuda_cores"])
def test_prefill_fused_combine_matches_unfused(tiny, cuda_cores):
    x = syn.activations(0, 0, 40, 512, stream=2)
    a = run_layer(tiny, x, cuda_cores=cuda_cores)
    b = run_layer(tiny, x, fused_prefill=True, cuda_cores=cuda_cores)
    np.testing.assert_array_equal(a["y"], b["y"])


# ---------------------------------------------------------------------------- routing edge cases

def route_only(wl, x_bits, bias=None):
    T = x_bits.shape[0]
    layer = MoeLayer(wl.d, wl.f, wl.E, wl.k, max(T, 1), wl.arena)
    b = None if bias is None else torch.from_numpy(bias).to(DEV)
    layer.route(bits_to_torch(x_bits, DEV), bits_to_torch(wl.wr, DEV), torch.from_numpy(wl.table).to(DEV), b)
    torch.cuda.synchronize()
    return dict(ids=layer.ids[:T].cpu().numpy(), w=layer.w[:T].cpu().numpy(), slots=layer.slots[:T].cpu().numpy(),
                status=int(layer.status.item()))


def check_route(wl, x_bits, got, bias=None):
    r = oracle.route_topk(x_bits, wl.wr, bias, wl.table, wl.k)
    np.testing.assert_array_equal(got["ids"], r["ids"])
    np.testing.assert_array_equal(got["slots"], r["slots"])
    np.testing.assert_allclose(got["w"], r["weights"], rtol=2e-5, atol=1e-7)


# T = 1, 5 and 16 take the decode router (one warp per expert, compensated logits, the
# last block selects); T = 24 the tiled router.
@pytest.mark.parametrize("T", [1, 5, 16, 24])
def test_router_ties_mask_bias_and_few_resident(T):
    d, E, k = 256, 40, 4
    wl = make_workload(d, 256, E, k, seed=5, scale=(-8, -4))
    wr = wl.wr.copy()
    wr[7] = wr[3]          # exact ties between experts 3, 7 and 21
    wr[21] = wr[3]
    wl.wr = wr
    x = syn.activations(5, 0, T, d)
    got = run_layer(wl, x)
    check_tokens(wl, x, got, list(range(T)))
    bias = syn.zipf_score_bias(5, 0, E, 1.2, 0.5)
    got = run_layer(wl, x, bias=bias)
    check_tokens(wl, x, got, list(range(T)), bias=bias)
    # keep-set mask: half the experts have no slot
    tab = wl.table.copy()
    tab[::2] = -1
    wl.table = tab
    got = run_layer(wl, x)
    assert np.all(got["ids"] % 2 == 1)
    check_tokens(wl, x, got, list(range(T)))
    # fewer than k resident
    tab = np.full(E, -1, np.int32)
    tab[[5, 9]] = [5, 9]
    wl.table = tab
    got = run_layer(wl, x[:2])
    assert got["status"] & moe.MOE_STATUS_FEW_RESIDENT
    assert got["ids"].tolist() == [[5, 9, -1, -1]] * min(T, 2)
    r = oracle.route_topk(x[:2], wl.wr, None, tab, k)
    np.testing.assert_array_equal(got["ids"], r["ids"])
    np.testing.assert_allclose(got["w"], r["weights"], rtol=2e-5)


@pytest.mark.parametrize("T", [1, 3, 8, 16, 40])
def test_router_wide_dynamic_range_and_saturation(T):
    """Activations scaled by 2^u, u uniform in [-24, 24] per element: logits span many
    orders of magnitude, most scores saturate to exactly 0 or 1 (ties broken by id), and
    the fast logit's error bound is exercised far from the N(0, 1) regime."""
    d, E, k = 1024, 200, 6
    wl = make_workload(d, 256, E, k, seed=11, table="permuted", scale=(-8, -4))
    x = syn.bf16_bits_to_f32(syn.activations(11, 0, T, d)).astype(np.float64)
    u = np.random.default_rng(11).integers(-24, 25, size=x.shape)
    xb = syn.f32_to_bf16_bits(np.ldexp(x, u).astype(np.float32))
    got = route_only(wl, xb)
    check_route(wl, xb, got)
    # moderate scale: scores spread over (0, 1) with close neighbours
    xb2 = syn.f32_to_bf16_bits((x * 3.0).astype(np.float32))
    bias = syn.zipf_score_bias(11, 0, E, 1.0, 1e-3)
    got = route_only(wl, xb2, bias=bias)
    check_route(wl, xb2, got, bias=bias)


def test_router_cancellation_of_large_products():
    """Each token carries +-2^20 at elements 0/1 (one lane's chunk) and 16/24 (two lanes),
    against equal router weights, so those products cancel exactly in the true logit while
    an uncompensated fp32 chain holding them loses the bits of every small product."""
    d, E, k, T = 512, 64, 4, 6
    wl = make_workload(d, 256, E, k, seed=12, scale=(-8, -4))
    x = syn.bf16_bits_to_f32(syn.activations(12, 0, T, d)).copy()
    big = np.float32(2.0 ** 20)
    x[:, 0], x[:, 1], x[:, 16], x[:, 24] = big, -big, big, -big
    w = syn.bf16_bits_to_f32(wl.wr).copy()
    w[:, 1] = w[:, 0]
    w[:, 24] = w[:, 16]
    wl.wr = syn.f32_to_bf16_bits(w)
    xb = syn.f32_to_bf16_bits(x)
    for n in (1, T):
        got = route_only(wl, xb[:n])
        check_route(wl, xb[:n], got)


def test_router_large_batch_bit_exact_ids():
    """Tiled router path (T > 16) with a skewing bias: every token's ids and slots."""
    d, E, k, T = 1024, 96, 6, 300
    wl = make_workload(d, 256, E, k, seed=2, table="permuted", scale=(-10, -6))
    bias = syn.zipf_score_bias(2, 0, E, 1.2, 0.04)
    x = syn.activations(2, 0, T, d)
    got = run_layer(wl, x, bias=bias)
    r = oracle.route_topk(x, wl.wr, bias, wl.table, k)
    np.testing.assert_array_equal(got["ids"], r["ids"])
    np.testing.assert_array_equal(got["slots"], r["slots"])
    np.testing.assert_allclose(got["w"], r["weights"], rtol=2e-5, atol=1e-7)


def test_bad_slot_is_reported_and_skipped():
    d, E, k = 256, 8, 2
    wl = make_workload(d, 256, E, k, seed=6, num_slots=8)
    tab = wl.table.copy()
    tab[:] = 100                # every slot outside the arena
    wl.table = tab
    x = syn.activations(6, 0, 2, d)
    got = run_layer(wl, x)
    assert got["status"] & moe.MOE_STATUS_BAD_SLOT
    assert np.all(got["y"] == 0)


def test_zero_tokens_is_a_no_op(tiny):
    layer = MoeLayer(512, 256, 16, 2, 4, tiny.arena)
    x = torch.zeros((0, 512), dtype=torch.bfloat16, device=DEV)
    moe.moe_route_topk(layer.dims, 0, layer.y, bits_to_torch(tiny.wr, DEV), None,
                       torch.from_numpy(tiny.table).to(DEV), layer.ids, layer.w, layer.slots, layer.status, layer.ws)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    del x


# ---------------------------------------------------------------------------- pages' shape

@pytest.fixture(scope="module")
def full_decode():
    """d=5120, f=2304, E=384, k=6, all experts resident behind a permuted slot table."""
    return make_workload(5120, 2304, 384, 6, seed=0, table="permuted", scale=(-10, -6))


@pytest.mark.parametrize("cuda_cores", [False, True], ids=["tensor_cores", "cuda_cores"])
def test_full_shape_decode_T1_sampled_tokens(full_decode, cuda_cores):
    wl = full_decode
    x = syn.activations(0, 0, 6, 5120, stream=3)
    for t in range(3):
        got = run_layer(wl, x[t:t + 1], cuda_cores=cuda_cores)
        check_tokens(wl, x[t:t + 1], got, [0])


@pytest.mark.parametrize("cuda_cores", [False, True], ids=["tensor_cores", "cuda_cores"])
def test_full_shape_verify_T16(full_decode, cuda_cores):
    wl = full_decode
    x = syn.activations(0, 0, 16, 5120, stream=4)
    got = run_layer(wl, x, cuda_cores=cuda_cores)
    check_tokens(wl, x, got, [0, 7, 15])


def assert_rows_equal_single_calls(wl, x, cuda_cores):
    """Each row of one call on all of x equals the call on that token alone, bit for bit."""
    big = run_layer(wl, x, cuda_cores=cuda_cores)
    assert big["status"] == 0
    for t in range(x.shape[0]):
        one = run_layer(wl, x[t:t + 1], cuda_cores=cuda_cores)
        assert one["status"] == 0
        np.testing.assert_array_equal(one["ids"][0], big["ids"][t])
        np.testing.assert_array_equal(one["slots"][0], big["slots"][t])
        assert one["w"][0].tobytes() == big["w"][t].tobytes(), t
        assert one["y"][0].tobytes() == big["y"][t].tobytes(), t   # fp32 view of the bf16 row
    return big


@pytest.mark.parametrize("cuda_cores", [False, True], ids=["tensor_cores", "cuda_cores"])
def test_verify_rows_equal_decode_calls(full_decode, cuda_cores):
    """DSpark verify: every row of a T=16 call reproduces the T=1 decode call on that token bit
    for bit (routing and output), including a token that appears twice."""
    x = syn.activations(0, 0, 16, 5120, stream=11).copy()
    x[9] = x[2]
    assert_rows_equal_single_calls(full_decode, x, cuda_cores)


def test_slots_shared_by_experts_and_split_keys():
    """16 experts on 3 slots: a token may route two of its experts to one slot, and at T=16 a
    slot collects more than 16 pairs, so its pairs form several keys.  Output against the
    oracle, and rows against single-token calls bit for bit."""
    wl = make_workload(1024, 768, 16, 4, seed=7, scale=(-9, -5), table=np.arange(16) % 3)
    x = syn.activations(7, 0, 16, 1024)
    big = assert_rows_equal_single_calls(wl, x, False)
    check_tokens(wl, x, big, list(range(16)))


def host_device_pointer(t):
    """Device address of pinned host tensor t (cudaHostGetDevicePointer)."""
    import ctypes
    rt = None
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
            break
        except OSError:
            pass
    if rt is None:
        return t.data_ptr()   # unified addressing: the host address is the device address
    dp = ctypes.c_void_p()
    assert rt.cudaHostGetDevicePointer(ctypes.byref(dp), ctypes.c_void_p(t.data_ptr()), 0) == 0
    return dp.value


@pytest.mark.parametrize("T", [3, 40])
def test_two_wave_moe_equals_one_wave(T):
    """Partial residency: with half the experts on hand, wave 1 computes their rows,
    one kernel gathers the missing experts from pinned host memory into their slots, wave 2
    computes the rest, and the fixed-order combine gives the one-wave result bit for bit."""
    d, f, E, k = 1024, 768, 16, 4
    full = make_workload(d, f, E, k, seed=21, scale=(-9, -5))        # identity table: slot e = expert e
    dims = moe.moe_dims(d, f, E, k)
    sb = moe.moe_slot_bytes(dims)
    store = torch.empty(E * sb, dtype=torch.uint8, pin_memory=True)  # every expert's slot image
    store.copy_(full.arena.buf[:E * sb].cpu())
    part = Arena(dims, E, DEV)
    part.buf.zero_()
    resident = torch.full((E,), -1, dtype=torch.int32, device=DEV)
    for e in (0, 2, 3, 5, 7, 8, 11, 13):
        part.buf[e * sb:(e + 1) * sb].copy_(full.arena.buf[e * sb:(e + 1) * sb])
        resident[e] = e
    x_bits = syn.activations(21, 0, T, d)
    x = bits_to_torch(x_bits, DEV)
    wr = bits_to_torch(full.wr, DEV)
    tab = torch.from_numpy(full.table).to(DEV)
    layer = MoeLayer(d, f, E, k, T, part)
    layer.route(x, wr, tab)
    n = T * k
    moe.moe_permute(dims, T, layer.ids, layer.offsets, layer.row_src, layer.row_dst, layer.ws)
    w1, w2, missing = (torch.empty(n, dtype=torch.int32, device=DEV) for _ in range(3))
    n_missing = torch.zeros(1, dtype=torch.int32, device=DEV)
    moe.moe_split_waves(dims, T, layer.ids, layer.slots, resident, E, w1, w2, missing, n_missing)
    rows = torch.full((n, d), float("nan"), dtype=torch.float32, device=DEV)
    ffn = lambda arena, slots, out: moe.moe_expert_ffn_fp4(
        dims, arena.c, T, x, layer.ids, slots, layer.w, layer.offsets, layer.row_src, layer.row_dst, 0, out, None,
        layer.status, layer.ws)
    ffn(part, w1, rows)
    moe.moe_gather_experts(dims, part.c, host_device_pointer(store), E, missing, n_missing, tab, resident, layer.status)
    ffn(part, w2, rows)
    y2 = torch.empty((T, d), dtype=torch.bfloat16, device=DEV)
    moe.moe_combine(dims, T, rows, layer.row_dst, layer.w, y2)
    rows1 = torch.empty_like(rows)
    ffn(full.arena, layer.slots, rows1)
    y1 = torch.empty_like(y2)
    moe.moe_combine(dims, T, rows1, layer.row_dst, layer.w, y1)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    ids = layer.ids[:T].cpu().numpy()
    want = sorted(set(int(e) for e in ids.ravel() if e >= 0) - {0, 2, 3, 5, 7, 8, 11, 13})
    assert int(n_missing.item()) == len(want) and missing[:len(want)].cpu().tolist() == want
    w1h, w2h, slots = w1.cpu().numpy(), w2.cpu().numpy(), layer.slots[:T].cpu().numpy().ravel()
    assert ((w1h >= 0) != (w2h >= 0)).all() and (np.maximum(w1h, w2h) == slots).all()
    for e in want:                                                   # gathered images and residency
        assert torch.equal(part.buf[e * sb:(e + 1) * sb], full.arena.buf[e * sb:(e + 1) * sb]), e
        assert int(resident[e].item()) == e
    valid = layer.row_src[:n].cpu().numpy() >= 0
    assert torch.equal(rows[torch.from_numpy(valid).to(DEV)].view(torch.int32),
                       rows1[torch.from_numpy(valid).to(DEV)].view(torch.int32))
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    check_tokens(full, x_bits, dict(ids=ids, slots=layer.slots[:T].cpu().numpy(), w=layer.w[:T].cpu().numpy(),
                                    y=y2.float().cpu().numpy()), list(range(min(T, 8))))


@pytest.mark.parametrize("T", [3, 40])
def test_cache_conditional_routing_two_waves(T):
    """Cache-conditional routing on a partly resident arena: moe_residency_bias gives
    the oracle's bias bit for bit, the router never masks (every expert keeps its slot), it
    picks resident experts more often than exact routing yet still picks some missing ones, and
    the two-wave layer (wave 1, gather, wave 2, fixed-order combine) matches the oracle layer
    routed with the same bias."""
    d, f, E, k, lam = 1024, 768, 16, 4, 0.05
    on = (1, 4, 6, 9, 10, 14)
    full = make_workload(d, f, E, k, seed=23, scale=(-9, -5))        # identity table
    dims = moe.moe_dims(d, f, E, k)
    sb = moe.moe_slot_bytes(dims)
    store = torch.empty(E * sb, dtype=torch.uint8, pin_memory=True)
    store.copy_(full.arena.buf[:E * sb].cpu())
    part = Arena(dims, E, DEV)
    part.buf.zero_()
    resident = torch.full((E,), -1, dtype=torch.int32, device=DEV)
    for e in on:
        part.buf[e * sb:(e + 1) * sb].copy_(full.arena.buf[e * sb:(e + 1) * sb])
        resident[e] = e
    res_host = resident.cpu().numpy()
    tab = torch.from_numpy(full.table).to(DEV)
    base = syn.zipf_score_bias(0, 0, E, 1.2, 0.01)
    bias = torch.empty(E, dtype=torch.float32, device=DEV)
    moe.moe_residency_bias(dims, torch.from_numpy(base).to(DEV), tab, resident, E, lam, bias)
    x_bits = syn.activations(23, 0, T, d)
    x = bits_to_torch(x_bits, DEV)
    layer = MoeLayer(d, f, E, k, T, part)
    layer.route(x, bits_to_torch(full.wr, DEV), tab, bias)
    n = T * k
    moe.moe_permute(dims, T, layer.ids, layer.offsets, layer.row_src, layer.row_dst, layer.ws)
    w1, w2, missing = (torch.empty(n, dtype=torch.int32, device=DEV) for _ in range(3))
    n_missing = torch.zeros(1, dtype=torch.int32, device=DEV)
    moe.moe_split_waves(dims, T, layer.ids, layer.slots, resident, E, w1, w2, missing, n_missing)
    rows = torch.full((n, d), float("nan"), dtype=torch.float32, device=DEV)
    ffn = lambda slots: moe.moe_expert_ffn_fp4(
        dims, part.c, T, x, layer.ids, slots, layer.w, layer.offsets, layer.row_src, layer.row_dst, 0, rows, None,
        layer.status, layer.ws)
    ffn(w1)
    moe.moe_gather_experts(dims, part.c, host_device_pointer(store), E, missing, n_missing, tab, resident, layer.status)
    ffn(w2)
    y = torch.empty((T, d), dtype=torch.bfloat16, device=DEV)
    moe.moe_combine(dims, T, rows, layer.row_dst, layer.w, y)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    want_bias = oracle.residency_bias(base, full.table, res_host, lam)
    np.testing.assert_array_equal(bias.cpu().numpy().view(np.int32), want_bias.view(np.int32))
    ids = layer.ids[:T].cpu().numpy()
    exact = oracle.route_topk(x_bits, full.wr, base, full.table, k)
    share = lambda a: np.isin(a, on).mean()
    assert share(ids) > share(exact["ids"]) and share(ids) < 1.0, (share(ids), share(exact["ids"]))
    got = dict(ids=ids, slots=layer.slots[:T].cpu().numpy(), w=layer.w[:T].cpu().numpy(), y=y.float().cpu().numpy())
    r = oracle.route_topk(x_bits, full.wr, want_bias, full.table, k)
    np.testing.assert_array_equal(got["ids"], r["ids"])
    np.testing.assert_array_equal(got["slots"], r["slots"])
    check_tokens(full, x_bits, got, list(range(min(T, 8))), bias=want_bias)


@pytest.mark.parametrize("cuda_cores", [False, True], ids=["tensor_cores", "cuda_cores"])
def test_full_shape_prefill_sampled_tokens(full_decode, cuda_cores):
    wl = full_decode
    T = 512
    bias = syn.zipf_score_bias(0, 0, 384, 1.2, 0.04)
    x = syn.activations(0, 0, T, 5120, stream=5)
    got = run_layer(wl, x, bias=bias, cuda_cores=cuda_cores)
    check_tokens(wl, x, got, [0, 1, 255, 511], bias=bias)


@pytest.mark.parametrize("fused", [False, True], ids=["rows_then_combine", "fused_combine"])
def test_config3_prefill_chunk_T4096(full_decode, fused):
    """The prefill chunk at the pages' shape (T = 4096, Zipf(1.2) bias, every expert resident):
    ids and slots of sampled tokens against the oracle router, the whole permutation against
    the oracle's permutation of the returned ids (bit for bit), sampled outputs against the
    oracle layer, and the skew the workload is meant to have (some experts get no token)."""
    wl = full_decode
    T = 4096
    bias = syn.zipf_score_bias(0, 0, 384, 1.2, 0.04)
    x = syn.activations(0, 0, T, 5120, stream=9)
    got = run_layer(wl, x, bias=bias, fused_prefill=fused)
    ids = got["ids"]
    assert got["status"] == 0
    counts = np.bincount(ids[ids >= 0], minlength=wl.E)
    assert (counts == 0).sum() >= 1 and counts.max() > 6 * T / wl.E
    perm = oracle.permute(ids, wl.E)
    np.testing.assert_array_equal(got["offsets"], perm["offsets"])
    n = perm["rows"]
    np.testing.assert_array_equal(got["row_src"][:n], perm["row_src"])
    np.testing.assert_array_equal(got["row_dst"], perm["row_dst"])
    check_tokens(wl, x, got, [0, 1, 2047, 4095], bias=bias)
    sample = np.random.default_rng(3).choice(T, 48, replace=False)
    r = oracle.route_topk(x[sample], wl.wr, bias, wl.table, wl.k)
    np.testing.assert_array_equal(ids[sample], r["ids"])
    np.testing.assert_array_equal(got["slots"][sample], r["slots"])
