"""cb3 expert format on the GPU against the oracle: the packer bit for bit (levels and every
3-bit index, read back through the documented slot layout), the cb3 decode FFN within the
output tolerance, multi-row calls equal to single-token calls, and the packer's flagged rows."""
import numpy as np
import pytest
import torch

import fp4_routed_expert_gb300 as moe
from fp4_routed_expert_gb300.layer import Arena, Cb3Arena, MoeLayer
import oracle
from synth import tensors as syn

from workloads import bits_to_torch, make_workload, row_rel_err

pytestmark = pytest.mark.gpu

TOL = 1e-2
DEV = "cuda"
ZQ = (2, 3, 0, 1)      # bit of element j's high index bit inside its nibble, by quarter j // 8


def cb3_decode_slot(buf: np.ndarray, d: int, f: int) -> dict:
    """Levels [rows, 8] (bf16 bits) and indices [rows, K] of one cb3 slot image, read by the
    layout the header and the kernel source state: levels 16 bytes per row (gate, up, down
    rows), then per row three arrays A, B, Z of K/32 words."""
    R = 2 * f + d
    lv = buf[:16 * R].view(np.uint16).reshape(R, 8)

    def rows(off, n, K):
        nc = K // 32
        w = buf[off:off + n * 3 * nc * 4].view(np.uint32).reshape(n, 3, nc)
        A, B, Z = w[:, 0], w[:, 1], w[:, 2]
        idx = np.zeros((n, K), np.uint8)
        for j in range(32):
            jj = j % 16
            low = ((A if j < 16 else B) >> (4 * (jj % 8) + 2 * (jj // 8))) & 3
            high = (Z >> (4 * (j % 8) + ZQ[j // 8])) & 1
            idx[:, j::32] = (low | (high << 2)).astype(np.uint8)
        return idx

    g0 = 16 * R
    return {"gate_cb": lv[:f], "up_cb": lv[f:2 * f], "down_cb": lv[2 * f:],
            "gate_idx": rows(g0, f, d), "up_idx": rows(g0 + f * 3 * d // 8, f, d),
            "down_idx": rows(g0 + 2 * f * 3 * d // 8, d, f)}


def pack_all(wl) -> Cb3Arena:
    dims = moe.moe_dims(wl.d, wl.f, wl.E, wl.k)
    cb = Cb3Arena(dims, wl.arena.num_slots, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for s in range(wl.arena.num_slots):
        cb.pack_from(wl.arena, s, s, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return cb


def slot_image(cb: Cb3Arena, s: int) -> np.ndarray:
    return cb.buf[s * cb.slot_bytes:(s + 1) * cb.slot_bytes].cpu().numpy()


def assert_pack_equal(got: dict, want: dict):
    for m in ("gate", "up", "down"):
        np.testing.assert_array_equal(got[m + "_cb"], want[m + "_cb"], err_msg=m)
        np.testing.assert_array_equal(got[m + "_idx"], want[m + "_idx"], err_msg=m)


def run_cb3(wl, cb, x_bits):
    T = x_bits.shape[0]
    layer = MoeLayer(wl.d, wl.f, wl.E, wl.k, max(T, 1), wl.arena)
    x = bits_to_torch(x_bits, DEV)
    layer.route(x, bits_to_torch(wl.wr, DEV), torch.from_numpy(wl.table).to(DEV))
    y = layer.experts_cb3(cb, x, T=T)
    torch.cuda.synchronize()
    return dict(ids=layer.ids[:T].cpu().numpy(), slots=layer.slots[:T].cpu().numpy(), status=int(layer.status.item()),
                y=y[:T].float().cpu().numpy(), y_bits=y[:T].view(torch.int16).cpu().numpy())


def check_cb3_tokens(wl, x_bits, got, tokens, packed: dict):
    """Oracle routing, oracle cb3 packing of the chosen slots, oracle cb3 FFN and combine."""
    r = oracle.route_topk(x_bits[tokens], wl.wr, None, wl.table, wl.k)
    np.testing.assert_array_equal(got["ids"][tokens], r["ids"])
    np.testing.assert_array_equal(got["slots"][tokens], r["slots"])
    ys = []
    for n, t in enumerate(tokens):
        z = np.zeros((wl.k, wl.d))
        for j in range(wl.k):
            s = int(r["slots"][n, j])
            if s not in packed:
                packed[s] = oracle.cb3_pack_expert(wl.expert_tensors(s))
            z[j] = oracle.cb3_expert_ffn(x_bits[t], packed[s])[1]
        ys.append(oracle.combine(z, r["weights"][n]))
    err = row_rel_err(got["y"][tokens], np.stack(ys))
    print("cb3 max row error %.3e over %d tokens" % (err.max(), len(tokens)))
    assert err.max() <= TOL, err


@pytest.fixture(scope="module")
def small_cb3():
    wl = make_workload(512, 256, 16, 4, seed=41, scale=(-9, -5), table="permuted")
    return wl, pack_all(wl), {}


def test_cb3_pack_matches_oracle(small_cb3):
    wl, cb, packed = small_cb3
    for s in range(wl.arena.num_slots):
        want = oracle.cb3_pack_expert(wl.expert_tensors(s))
        packed[s] = want
        assert_pack_equal(cb3_decode_slot(slot_image(cb, s), wl.d, wl.f), want)


@pytest.mark.parametrize("T", [1, 3, 16])
def test_cb3_ffn_matches_oracle(small_cb3, T):
    wl, cb, packed = small_cb3
    x = syn.activations(41, 0, T, wl.d)
    got = run_cb3(wl, cb, x)
    assert got["status"] == 0
    check_cb3_tokens(wl, x, got, list(range(T)), packed)


def test_cb3_prefill_chunk_in_16_token_calls(small_cb3):
    """T = 40 (a prefill-size call, the tiled router): the cb3 experts run as consecutive calls
    of 16 tokens; sampled tokens against the oracle, and every row equal to the T = 1 call on
    that token bit for bit."""
    wl, cb, packed = small_cb3
    x = syn.activations(41, 0, 40, wl.d, stream=6)
    got = run_cb3(wl, cb, x)
    assert got["status"] == 0
    check_cb3_tokens(wl, x, got, [0, 15, 16, 39], packed)
    for t in (0, 17, 39):
        one = run_cb3(wl, cb, x[t:t + 1])
        np.testing.assert_array_equal(one["ids"][0], got["ids"][t])
        np.testing.assert_array_equal(got["y_bits"][t], one["y_bits"][0], err_msg=str(t))


def test_cb3_rows_equal_decode_calls(small_cb3):
    wl, cb, _ = small_cb3
    x = syn.activations(41, 0, 16, wl.d, stream=2)
    many = run_cb3(wl, cb, x)
    for t in range(16):
        one = run_cb3(wl, cb, x[t:t + 1])
        np.testing.assert_array_equal(many["y_bits"][t], one["y_bits"][0], err_msg=str(t))


@pytest.mark.parametrize("T", [1, 3, 16])
def test_cb3_two_waves_equal_one_wave(small_cb3, T):
    """cb3 slots in the two-wave flow: rows of the experts on hand (moe_expert_ffn_cb3_rows with
    the wave-1 slots), the missing cb3 slot images gathered from pinned host memory, rows of the
    rest, then moe_combine: equal bit for bit to moe_expert_ffn_cb3 on the fully resident cb3
    arena, and every row equal to the one-wave rows."""
    from test_gpu_parity import host_device_pointer
    wl, cb, _ = small_cb3
    dims = moe.moe_dims(wl.d, wl.f, wl.E, wl.k)
    sb, ns = cb.slot_bytes, wl.arena.num_slots
    store = torch.empty(wl.E * sb, dtype=torch.uint8, pin_memory=True)   # expert e's cb3 image at e * sb
    for e in range(wl.E):
        s = int(wl.table[e])
        store[e * sb:(e + 1) * sb].copy_(cb.buf[s * sb:(s + 1) * sb].cpu())
    part = Cb3Arena(dims, ns, DEV)
    part.buf.zero_()
    resident = torch.full((ns,), -1, dtype=torch.int32, device=DEV)
    on_hand = (0, 2, 3, 5, 7, 8, 11, 13)
    for e in on_hand:
        s = int(wl.table[e])
        part.buf[s * sb:(s + 1) * sb].copy_(cb.buf[s * sb:(s + 1) * sb])
        resident[s] = e
    x_bits = syn.activations(41, 0, T, wl.d, stream=5)
    x = bits_to_torch(x_bits, DEV)
    tab = torch.from_numpy(wl.table).to(DEV)
    layer = MoeLayer(wl.d, wl.f, wl.E, wl.k, T, wl.arena)
    layer.route(x, bits_to_torch(wl.wr, DEV), tab)
    n = T * wl.k
    moe.moe_permute(dims, T, layer.ids, layer.offsets, layer.row_src, layer.row_dst, layer.ws)
    w1, w2, missing = (torch.empty(n, dtype=torch.int32, device=DEV) for _ in range(3))
    n_missing = torch.zeros(1, dtype=torch.int32, device=DEV)
    moe.moe_split_waves(dims, T, layer.ids, layer.slots, resident, ns, w1, w2, missing, n_missing)
    rows = torch.full((n, wl.d), float("nan"), dtype=torch.float32, device=DEV)
    moe.moe_expert_ffn_cb3_rows(dims, part.c, T, x, w1, layer.row_dst, rows, layer.status, layer.ws)
    moe.moe_gather_experts(dims, part.c, host_device_pointer(store), wl.E, missing, n_missing, tab, resident,
                           layer.status)
    moe.moe_expert_ffn_cb3_rows(dims, part.c, T, x, w2, layer.row_dst, rows, layer.status, layer.ws)
    y2 = torch.empty((T, wl.d), dtype=torch.bfloat16, device=DEV)
    moe.moe_combine(dims, T, rows, layer.row_dst, layer.w, y2)
    rows1 = torch.full_like(rows, float("nan"))
    moe.moe_expert_ffn_cb3_rows(dims, cb.c, T, x, layer.slots, layer.row_dst, rows1, layer.status, layer.ws)
    y1 = layer.experts_cb3(cb, x, T=T)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    ids = layer.ids[:T].cpu().numpy()
    want = sorted(set(int(e) for e in ids.ravel() if e >= 0) - set(on_hand))
    assert int(n_missing.item()) == len(want) and missing[:len(want)].cpu().tolist() == want
    valid = torch.from_numpy(layer.row_src[:n].cpu().numpy() >= 0).to(DEV)
    assert torch.equal(rows[valid].view(torch.int32), rows1[valid].view(torch.int32))
    assert torch.equal(y1[:T].view(torch.int16), y2.view(torch.int16))


def test_cb3_zero_tokens_and_bad_slot(small_cb3):
    wl, cb, _ = small_cb3
    dims = moe.moe_dims(wl.d, wl.f, wl.E, wl.k)
    layer = MoeLayer(wl.d, wl.f, wl.E, wl.k, 2, wl.arena)
    x = bits_to_torch(syn.activations(41, 0, 2, wl.d), DEV)
    y = torch.full((2, wl.d), 7.0, dtype=torch.bfloat16, device=DEV)
    launched = moe.moe_kernel_launches()
    moe.moe_expert_ffn_cb3(dims, cb.c, 0, x, layer.slots, layer.w, y, layer.status, layer.ws)
    assert moe.moe_kernel_launches() == launched
    layer.slots.copy_(torch.tensor([[0, 1, 2, 99], [3, 4, 5, 6]], dtype=torch.int32))
    layer.w.fill_(0.25)
    moe.moe_expert_ffn_cb3(dims, cb.c, 2, x, layer.slots, layer.w, y, layer.status, layer.ws)
    torch.cuda.synchronize()
    assert int(layer.status.item()) & moe.MOE_STATUS_BAD_SLOT
    assert torch.isfinite(y.float()).all()


def test_cb3_flags_unpackable_rows():
    """d = 5120, f = 256: gate row 0 gets 160 distinct scale bytes (over 256 distinct values)
    and down row 3 a NaN scale; both are written as zero and flagged, every other row equals
    the oracle's packing."""
    d, f = 5120, 256
    dims = moe.moe_dims(d, f, 4, 2)
    t = syn.expert_tensors(7, 0, 0, d, f, -8, -4)
    t["gate_s"] = t["gate_s"].copy()
    t["gate_s"][0] = np.arange(20, 180, dtype=np.uint8)
    t["down_s"] = t["down_s"].copy()
    t["down_s"][3, 2] = 255
    fp4 = Arena(dims, 1, DEV)
    dev = {n: torch.from_numpy(np.ascontiguousarray(v)).to(DEV) for n, v in t.items()}
    fp4.pack(0, dev)
    cb = Cb3Arena(dims, 1, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    cb.pack_from(fp4, 0, 0, st)
    torch.cuda.synchronize()
    assert int(st.item()) == moe.MOE_STATUS_CB3_ROW
    got = cb3_decode_slot(slot_image(cb, 0), d, f)
    assert not got["gate_cb"][0].any() and not got["gate_idx"][0].any()
    assert not got["down_cb"][3].any() and not got["down_idx"][3].any()
    ok = dict(t)
    ok["gate_s"] = t["gate_s"].copy()
    ok["gate_s"][0] = 127
    ok["down_s"] = t["down_s"].copy()
    ok["down_s"][3] = 127
    want = oracle.cb3_pack_expert(ok)
    for m, bad in (("gate", 0), ("down", 3)):
        keep = np.arange(got[m + "_cb"].shape[0]) != bad
        np.testing.assert_array_equal(got[m + "_cb"][keep], want[m + "_cb"][keep])
        np.testing.assert_array_equal(got[m + "_idx"][keep], want[m + "_idx"][keep])
    np.testing.assert_array_equal(got["up_cb"], want["up_cb"])
    np.testing.assert_array_equal(got["up_idx"], want["up_idx"])


def test_cb3_full_shape_decode_T1():
    """d = 5120, f = 2304, k = 6 (16 experts, permuted slots): one token through the cb3 path
    against the oracle, and the six chosen slots' packing bit for bit."""
    wl = make_workload(5120, 2304, 16, 6, seed=3, scale=(-10, -6), table="permuted")
    cb = pack_all(wl)
    x = syn.activations(3, 0, 1, 5120, stream=4)
    got = run_cb3(wl, cb, x)
    assert got["status"] == 0
    packed = {}
    check_cb3_tokens(wl, x, got, [0], packed)
    for s, want in packed.items():
        assert_pack_equal(cb3_decode_slot(slot_image(cb, s), wl.d, wl.f), want)
