"""Pins for the CPU oracle: each test checks an oracle function against something other
than the oracle itself -- a bit-field definition, a library conversion, exact rational
arithmetic, multi-precision evaluation, brute force, a closed form, a hand-worked fixture,
or an independent fp64 re-derivation written here.  No GPU is involved."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from synth import tensors as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- helpers

def e2m1_from_bits(code):
    """e2m1 from its fields: sign, 2-bit exponent with bias 1, 1 mantissa bit."""
    s, e, m = code >> 3, (code >> 1) & 3, code & 1
    mag = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
    return -mag if s else mag


def bf16_exact(bits):
    """Exact rational value of a finite bf16 bit pattern, from its fields."""
    s, e, m = bits >> 15, (bits >> 7) & 0xFF, bits & 0x7F
    v = Fraction(m, 128) * Fraction(2) ** -126 if e == 0 else (1 + Fraction(m, 128)) * Fraction(2) ** (e - 127)
    return -v if s else v


def round_fraction_to_f32(v: Fraction) -> np.float32:
    """Round an exact rational to the nearest fp32 (ties to even), by integer arithmetic."""
    if v == 0:
        return np.float32(0.0)
    neg = v < 0
    a = -v if neg else v
    # find e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    q = max(e - 23, -149)                 # quantum exponent
    scaled = a / Fraction(2) ** q
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    val = n * (2.0 ** q) if q >= -1074 else 0.0
    r = np.float32(val) if val < 2.0 ** 128 else np.float32(np.inf)
    return -r if neg else r


def random_bf16(rng, n, lo_exp=-30, hi_exp=10):
    """bf16 bit patterns with exponents spread over [lo_exp, hi_exp] and random signs."""
    e = rng.integers(lo_exp, hi_exp + 1, n) + 127
    e = np.clip(e, 0, 254)
    m = rng.integers(0, 128, n)
    s = rng.integers(0, 2, n)
    return ((s << 15) | (e << 7) | m).astype(np.uint16)


def decode_matrix(q, s):
    """Independent numpy decode of a canonical [rows, K/2] code matrix and [rows, K/32]
    scale matrix into fp64, from the e2m1 and UE8M0 bit-field definitions."""
    q = np.asarray(q, np.uint8)
    rows, half = q.shape
    codes = np.empty((rows, half * 2), np.int64)
    codes[:, 0::2] = q & 15
    codes[:, 1::2] = q >> 4
    table = np.array([e2m1_from_bits(c) for c in range(16)])
    scale = np.ldexp(1.0, np.asarray(s, np.int64) - 127)
    return table[codes] * np.repeat(scale, 32, axis=1)


def bf16_to_f64(b):
    return syn.bf16_bits_to_f32(b).astype(np.float64)


# ----------------------------------------------------------------------------- formats

def test_e2m1_table_matches_field_definition():
    for c in range(16):
        want = e2m1_from_bits(c)
        got = oracle.e2m1_value(c)
        assert got == want
        assert math.copysign(1.0, got) == math.copysign(1.0, want if c != 8 else -0.0)
    assert math.copysign(1.0, oracle.e2m1_value(8)) < 0  # code 8 is -0


def test_ue8m0_is_an_fp32_exponent_field():
    for b in range(1, 255):
        want = np.array([b << 23], np.uint32).view(np.float32)[0]
        assert oracle.ue8m0_value(b) == float(want)
    # byte 0 is 2^-127, the fp32 subnormal with only mantissa bit 22 set -- not zero
    assert oracle.ue8m0_value(0) == float(np.array([1 << 22], np.uint32).view(np.float32)[0])
    assert math.isnan(oracle.ue8m0_value(255))


def test_code_times_scale_brute_force():
    """All 16 codes x 255 finite scale bytes through the packed-row accessor."""
    import ctypes
    L = oracle.lib()
    for code in range(16):
        row = np.full(16, code | (code << 4), np.uint8)   # 32 codes
        for b in range(255):
            srow = np.array([b], np.uint8)
            got = L.oracle_weight_at(row.ctypes.data_as(ctypes.c_void_p),
                                     srow.ctypes.data_as(ctypes.c_void_p), 5)
            scale = float(np.array([b << 23 if b else 1 << 22], np.uint32).view(np.float32)[0])
            want = e2m1_from_bits(code) * scale
            assert got == want, (code, b)


def test_nibble_order_hand_packed():
    """Byte 0x21 holds codes (1, 2) = (0.5, 1.0); byte 0xF8 holds (8, 15) = (-0, -6)."""
    import ctypes
    L = oracle.lib()
    row = np.array([0x21, 0xF8], np.uint8)
    p = row.ctypes.data_as(ctypes.c_void_p)
    assert [L.oracle_code_at(p, k) for k in range(4)] == [1, 2, 8, 15]
    s = np.array([127], np.uint8)
    ps = s.ctypes.data_as(ctypes.c_void_p)
    assert [L.oracle_weight_at(p, ps, k) for k in range(4)] == [0.5, 1.0, -0.0, -6.0]


def test_bf16_decode_matches_torch_for_every_pattern():
    torch = pytest.importorskip("torch")
    bits = np.arange(65536, dtype=np.int64)
    finite = ((bits >> 7) & 0xFF) != 0xFF
    t = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    for b in bits[finite][::7]:
        assert oracle.bf16_value(int(b)) == t[b]


def test_bf16_rounding_from_double():
    rng = np.random.default_rng(1)
    vals = list(rng.normal(size=2000) * np.exp(rng.uniform(-60, 60, size=2000)))
    # exact ties: 1 + 2^-8 (tie, even -> 1), 1 + 3*2^-8 (tie, even -> 1 + 2^-6)
    vals += [1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 2.0 ** -134, 3 * 2.0 ** -135,
             2.0 ** -140, 3.4e38, 3.4e39, 0.0, -0.0]
    for v in vals:
        got = oracle.bf16_from_double(float(v))
        # independent: exact rational rounding with 8 significant bits, subnormal quantum 2^-133
        a = Fraction(abs(v))
        if a == 0:
            want = 0x8000 if math.copysign(1, v) < 0 else 0
        else:
            e = math.frexp(abs(v))[1] - 1
            q = max(e - 7, -133)
            n = a / Fraction(2) ** q
            fl = n.numerator // n.denominator
            rem = n - fl
            if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2):
                fl += 1
            r = Fraction(fl) * Fraction(2) ** q
            if r >= Fraction(2) ** 128:
                want = 0x7F80
            else:
                f32 = np.array([float(r)], np.float32).view(np.uint32)[0]
                want = int(f32 >> 16) & 0x7FFF
            if v < 0:
                want |= 0x8000
        assert got == want, v


# ----------------------------------------------------------------------------- exact logit

def test_dot_rn32_matches_exact_rational_sum():
    rng = np.random.default_rng(2)
    for trial in range(120):
        n = int(rng.integers(1, 200))
        lo = int(rng.integers(-140, 0))
        x = random_bf16(rng, n, lo, lo + int(rng.integers(0, 60)))
        w = random_bf16(rng, n, -40, 5)
        if trial % 5 == 4:          # bf16 subnormals against large partners
            x = random_bf16(rng, n, -160, -127)
            w = random_bf16(rng, n, 90, 126)
        if trial % 3 == 0:          # heavy cancellation
            w[: n // 2] = w[n // 2: 2 * (n // 2)] ^ 0x8000
            x[: n // 2] = x[n // 2: 2 * (n // 2)]
        exact = sum((bf16_exact(int(a)) * bf16_exact(int(b)) for a, b in zip(x, w)), Fraction(0))
        got, bad = oracle.dot_bf16_rn32(x, w)
        assert not bad
        want = round_fraction_to_f32(exact)
        assert got == want or (got == 0 and want == 0), (trial, got, want)


def bf16_of(v):
    return int(syn.f32_to_bf16_bits(np.array([v], np.float32))[0])


def test_dot_rn32_hand_midpoints():
    """Sums built to sit on or just beside an fp32 rounding midpoint."""
    one, t24, t60 = bf16_of(1.0), bf16_of(2.0 ** -24), bf16_of(2.0 ** -60)
    ones = [one] * 3
    # 1 + 2^-24 is exactly halfway between 1 and 1 + 2^-23: ties to even -> 1
    assert oracle.dot_bf16_rn32(np.array([one, t24], np.uint16), np.array(ones[:2], np.uint16))[0] == np.float32(1.0)
    # a 2^-60 term past the midpoint must round up -- an fp64 running sum would lose it
    v, _ = oracle.dot_bf16_rn32(np.array([one, t24, t60], np.uint16), np.array(ones, np.uint16))
    assert v == np.float32(1.0 + 2.0 ** -23)
    # the same term below the midpoint rounds down
    v, _ = oracle.dot_bf16_rn32(np.array([one, t24, t60 | 0x8000], np.uint16), np.array(ones, np.uint16))
    assert v == np.float32(1.0)
    # complete cancellation of huge terms leaves the small one exactly
    big = bf16_of(2.0 ** 100)
    v, _ = oracle.dot_bf16_rn32(np.array([big, bf16_of(3.0), big ^ 0x8000], np.uint16), np.array(ones, np.uint16))
    assert v == np.float32(3.0)
    # a bf16 subnormal (0x0003 = 3 * 2^-133) times 2^120 is exactly 3 * 2^-13
    v, _ = oracle.dot_bf16_rn32(np.array([3], np.uint16), np.array([bf16_of(2.0 ** 120)], np.uint16))
    assert v == np.float32(3 * 2.0 ** -13)
    # subnormal products: 2^-133 * 2^-133 = 2^-266 is far below fp32's 2^-149 -> 0
    tiny = 1  # bf16 subnormal 2^-133
    assert oracle.dot_bf16_rn32(np.array([tiny], np.uint16), np.array([tiny], np.uint16))[0] == 0
    # overflow beyond fp32 gives infinity
    huge = bf16_of(2.0 ** 127)
    v, _ = oracle.dot_bf16_rn32(np.array([huge, huge], np.uint16), np.array([bf16_of(4.0)] * 2, np.uint16))
    assert np.isinf(v) and v > 0
    # non-finite inputs are flagged
    _, bad = oracle.dot_bf16_rn32(np.array([0x7F80], np.uint16), np.array([one], np.uint16))
    assert bad


def test_router_score_is_correctly_rounded_sigmoid():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.prec = 200
    rng = np.random.default_rng(3)
    ls = np.concatenate([rng.normal(size=4000) * 3, rng.uniform(-110, 30, size=1000),
                         [0.0, -0.0, 1e-30, -1e-30, 20.0, 40.0, -80.0, -103.0, -104.0, -200.0]]).astype(np.float32)
    mism = 0
    for l in ls:
        got = oracle.router_score(l)
        exact = 1 / (1 + mpmath.exp(-mpmath.mpf(float(l))))
        want = round_fraction_to_f32(Fraction(int(exact.man)) * Fraction(2) ** int(exact.exp))
        if got != want:
            mism += 1
            assert abs(float(got) - float(want)) <= np.spacing(np.float32(want)), l
    assert mism == 0
    assert oracle.router_score(0.0) == np.float32(0.5)
    assert oracle.router_score(40.0) == np.float32(1.0)


# ----------------------------------------------------------------------------- router

def _golden_router_case(g, case):
    d, E = g["d"], g["E"]
    wr = np.stack([syn.f32_to_bf16_bits(np.full(d, c, np.float32)) for c in g["row_constants"]])
    x = syn.f32_to_bf16_bits(np.full((1, d), case["x"], np.float32))
    bias = None if case["bias"] is None else np.array(case["bias"], np.float32)
    return x, wr, bias, np.array(case["slots"], np.int32)


def test_router_hand_worked_cases():
    g = json.load(open(os.path.join(GOLDEN, "router_hand.json")))
    for case in g["cases"]:
        x, wr, bias, tab = _golden_router_case(g, case)
        r = oracle.route_topk(x, wr, bias, tab, g["k"])
        assert r["ids"][0].tolist() == case["ids"], case["name"]
        assert r["slots"][0].tolist() == case["out_slots"], case["name"]
        assert r["status"] == case["status"], case["name"]
        np.testing.assert_allclose(r["weights"][0], case["weights"], rtol=2e-7, atol=0, err_msg=case["name"])


def test_router_brute_force_tiny():
    """Independent restatement on random tiny inputs: exact rational logits, double sigmoid,
    python sort by (-key, id)."""
    rng = np.random.default_rng(4)
    for trial in range(25):
        T, d, E, k = 3, 64, 12, 3
        x = syn.f32_to_bf16_bits(rng.normal(size=(T, d)).astype(np.float32))
        wr = syn.f32_to_bf16_bits((rng.normal(size=(E, d)) * 0.05).astype(np.float32))
        if trial % 4 == 1:                      # forced exact ties between experts
            wr[5] = wr[2]
            wr[9] = wr[2]
        tab = np.arange(E, dtype=np.int32)
        if trial % 4 == 2:
            tab[rng.choice(E, 4, replace=False)] = -1
        bias = (rng.normal(size=E) * 0.05).astype(np.float32) if trial % 2 else None
        r = oracle.route_topk(x, wr, bias, tab, k)
        for t in range(T):
            keys = []
            s32 = {}
            for e in range(E):
                ex = sum((bf16_exact(int(a)) * bf16_exact(int(b)) for a, b in zip(x[t], wr[e])), Fraction(0))
                l32 = round_fraction_to_f32(ex)
                s = np.float32(1.0 / (1.0 + math.exp(-float(l32))))
                s32[e] = s
                key = np.float32(s + (bias[e] if bias is not None else np.float32(0)))
                if tab[e] >= 0:
                    keys.append((-float(key), e))
            chosen = sorted(e for _, e in sorted(keys)[:k])
            assert r["ids"][t].tolist() == chosen
            tot = np.float32(0)
            for e in chosen:
                tot = np.float32(tot + s32[e])
            np.testing.assert_array_equal(r["weights"][t], np.array([np.float32(s32[e] / tot) for e in chosen], np.float32))


# ----------------------------------------------------------------------------- permute

def test_permute_matches_stable_sort_and_invariants():
    rng = np.random.default_rng(5)
    for trial in range(30):
        T, k, E = int(rng.integers(1, 40)), int(rng.integers(1, 7)), int(rng.integers(1, 20))
        ids = rng.integers(-1, E, size=(T, k)).astype(np.int32)
        p = oracle.permute(ids, E)
        flat = [(int(ids[t, j]), t, j) for t in range(T) for j in range(k) if ids[t, j] >= 0]
        want = [t * k + j for (_, t, j) in sorted(flat)]
        assert p["row_src"].tolist() == want
        off = p["offsets"]
        assert off[0] == 0 and off[E] == len(want) and np.all(np.diff(off) >= 0)
        for e in range(E):
            assert off[e + 1] - off[e] == int((ids == e).sum())
        for r, src in enumerate(p["row_src"]):
            assert p["row_dst"][src] == r
        assert np.all(p["row_dst"][ids.reshape(-1) < 0] == -1)


# ----------------------------------------------------------------------------- FFN

def _expert(rng, d, f, lo=-8, hi=-4):
    return {
        "gate_q": rng.integers(0, 256, (f, d // 2), dtype=np.uint8),
        "gate_s": (127 + rng.integers(lo, hi + 1, (f, d // 32))).astype(np.uint8),
        "up_q": rng.integers(0, 256, (f, d // 2), dtype=np.uint8),
        "up_s": (127 + rng.integers(lo, hi + 1, (f, d // 32))).astype(np.uint8),
        "down_q": rng.integers(0, 256, (d, f // 2), dtype=np.uint8),
        "down_s": (127 + rng.integers(lo, hi + 1, (d, f // 32))).astype(np.uint8),
    }


def test_ffn_closed_form_all_ones():
    """Every weight 1.0 (code 2, scale byte 127): g = u = S = sum(x), h = silu(S) S,
    z_r = f h."""
    d, f = 64, 32
    ex = {n: np.full(s, 0x22 if n.endswith("_q") else 127, np.uint8)
          for n, s in syn.expert_tensor_shapes(d, f).items()}
    rng = np.random.default_rng(6)
    x = syn.f32_to_bf16_bits(rng.normal(size=d).astype(np.float32) * 0.1)
    S = float(np.sum(bf16_to_f64(x)))
    h, z = oracle.expert_ffn(x, ex)
    hs = S / (1 + math.exp(-S)) * S
    np.testing.assert_allclose(h, hs, rtol=1e-14)
    np.testing.assert_allclose(z, f * hs, rtol=1e-14)


def test_ffn_closed_form_diagonal():
    """W_gate = I (code 2), W_up = 2I (code 4), W_down = I: z = h = silu(x) * 2x."""
    d = f = 32
    eye = np.zeros((32, 32), np.int64)
    def pack(codes):
        return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    ex = {"gate_q": pack(np.eye(32, dtype=np.int64) * 2), "up_q": pack(np.eye(32, dtype=np.int64) * 4),
          "down_q": pack(np.eye(32, dtype=np.int64) * 2)}
    for n in ("gate_s", "up_s", "down_s"):
        ex[n] = np.full((32, 1), 127, np.uint8)
    x = syn.f32_to_bf16_bits(np.linspace(-3, 3, 32).astype(np.float32))
    xv = bf16_to_f64(x)
    h, z = oracle.expert_ffn(x, ex)
    want = xv / (1 + np.exp(-xv)) * 2 * xv
    np.testing.assert_allclose(h, want, rtol=1e-15, atol=1e-300)
    np.testing.assert_allclose(z, want, rtol=1e-15, atol=1e-300)
    del eye


def test_ffn_against_independent_numpy():
    rng = np.random.default_rng(7)
    d, f = 128, 64
    ex = _expert(rng, d, f)
    x = syn.f32_to_bf16_bits(rng.normal(size=d).astype(np.float32))
    h, z = oracle.expert_ffn(x, ex)
    xv = bf16_to_f64(x)
    g = decode_matrix(ex["gate_q"], ex["gate_s"]) @ xv
    u = decode_matrix(ex["up_q"], ex["up_s"]) @ xv
    hh = g * u / (1 + np.exp(-g))
    zz = decode_matrix(ex["down_q"], ex["down_s"]) @ hh
    np.testing.assert_allclose(h, hh, rtol=1e-12, atol=1e-12 * np.abs(hh).max())
    np.testing.assert_allclose(z, zz, rtol=1e-12, atol=1e-12 * np.abs(zz).max())


def test_combine_fixed_order_and_one_hot():
    rng = np.random.default_rng(8)
    z = rng.normal(size=(3, 16))
    y = oracle.combine(z, np.array([1.0, 0.0, 0.0], np.float32))
    np.testing.assert_array_equal(y, z[0])
    w = np.array([0.25, 0.5, 0.25], np.float32)
    y = oracle.combine(z, w)
    want = (0.25 * z[0] + 0.5 * z[1]) + 0.25 * z[2]
    np.testing.assert_array_equal(y, want)


# ----------------------------------------------------------------------------- FFN in fp32

U32 = 2.0 ** -24     # unit roundoff of fp32


def _exp_f32(v):
    """exp(v) for a float32 v, computed in double and rounded once to float32 (libm's expf
    may differ from this by one unit in the last place)."""
    return np.float32(math.exp(float(v)))


def _ffn_f32_numpy(x_bits, ex):
    """The fp32 FFN re-derived here from the bit-field decode: products exact (checked), every
    sum an explicit float32 accumulation in index order, vectorised over rows only."""
    xf = syn.bf16_bits_to_f32(x_bits)
    Wg = decode_matrix(ex["gate_q"], ex["gate_s"]).astype(np.float32)
    Wu = decode_matrix(ex["up_q"], ex["up_s"]).astype(np.float32)
    Wd = decode_matrix(ex["down_q"], ex["down_s"]).astype(np.float32)
    Pg, Pu = (Wg * xf[None, :]), (Wu * xf[None, :])
    assert np.array_equal(Pg.astype(np.float64), Wg.astype(np.float64) * xf.astype(np.float64)[None, :])  # exact
    g = np.zeros(Wg.shape[0], np.float32)
    u = np.zeros(Wg.shape[0], np.float32)
    for k in range(Wg.shape[1]):
        g = (g + Pg[:, k]).astype(np.float32)
        u = (u + Pu[:, k]).astype(np.float32)
    den = np.array([np.float32(1.0) + _exp_f32(-gi) for gi in g], np.float32)
    h = ((g / den).astype(np.float32) * u).astype(np.float32)
    z = np.zeros(Wd.shape[0], np.float32)
    for i in range(Wd.shape[1]):
        z = (z + (Wd[:, i] * h[i]).astype(np.float32)).astype(np.float32)
    return g, u, h, z


def test_ffn_f32_weights_are_exact():
    """code * 2^(b-127) in fp32 equals the bit-field value for every code and scale byte where
    that value is within the fp32 range, including b = 0 (the subnormal 2^-127), and is the
    signed infinity beyond it (codes 2..6 at b = 254 exceed the largest fp32)."""
    fmax = float(np.finfo(np.float32).max)
    for b in range(0, 255):
        for c in range(16):
            q = np.array([c | (c << 4)], np.uint8)
            s = np.array([b], np.uint8)
            want = e2m1_from_bits(c) * 2.0 ** (b - 127)
            if abs(want) > fmax:
                want = math.copysign(math.inf, want)
            assert float(oracle.weight_at_f32(q, s, 0)) == want
            assert float(oracle.weight_at_f32(q, s, 1)) == want


def test_ffn_f32_closed_form_all_ones():
    """Every weight 1.0 and x a set of multiples of 2^-8 whose partial sums are exact in fp32:
    g = u = S exactly; h = fp32 steps of silu(S) S; z = f copies of h summed in fp32."""
    d, f = 64, 32
    ex = {n: np.full(sh, 0x22 if n.endswith("_q") else 127, np.uint8)
          for n, sh in syn.expert_tensor_shapes(d, f).items()}
    rng = np.random.default_rng(16)
    xv = rng.integers(-40, 41, d).astype(np.float32) / 256.0
    x = syn.f32_to_bf16_bits(xv)
    S = np.float32(np.sum(xv.astype(np.float64)))          # exact: |partial sums| < 2^5, step 2^-8
    h, z = oracle.expert_ffn_f32(x, ex)
    den = np.float32(np.float32(1.0) + _exp_f32(-S))
    hs = np.float32(np.float32(S / den) * S)
    np.testing.assert_allclose(h, hs, rtol=3 * U32)        # expf within an ulp of exp
    zs = np.float32(0)
    for _ in range(f):
        zs = np.float32(zs + h[0])
    assert np.all(h == h[0]) and np.all(z == zs)


def test_ffn_f32_closed_form_diagonal():
    """W_gate = I, W_up = 2I, W_down = I: z_i = h_i = fp32(fp32(x_i / (1 + expf(-x_i))) * 2x_i)."""
    d = f = 32
    def pack(codes):
        return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    ex = {"gate_q": pack(np.eye(32, dtype=np.int64) * 2), "up_q": pack(np.eye(32, dtype=np.int64) * 4),
          "down_q": pack(np.eye(32, dtype=np.int64) * 2)}
    for n in ("gate_s", "up_s", "down_s"):
        ex[n] = np.full((32, 1), 127, np.uint8)
    xv = syn.bf16_bits_to_f32(syn.f32_to_bf16_bits(np.linspace(-3, 3, 32).astype(np.float32)))
    x = syn.f32_to_bf16_bits(xv)
    h, z = oracle.expert_ffn_f32(x, ex)
    want = np.array([np.float32(np.float32(v / np.float32(np.float32(1) + _exp_f32(-v))) * np.float32(2 * v))
                     for v in xv], np.float32)
    np.testing.assert_allclose(h, want, rtol=3 * U32, atol=0)
    np.testing.assert_array_equal(z, h)                     # one nonzero term per row: exact


def test_ffn_f32_against_independent_numpy_float32():
    rng = np.random.default_rng(17)
    d, f = 128, 64
    ex = _expert(rng, d, f)
    x = syn.f32_to_bf16_bits(rng.normal(size=d).astype(np.float32))
    h, z = oracle.expert_ffn_f32(x, ex)
    g, u, hh, zz = _ffn_f32_numpy(x, ex)
    # g and u are identical sequences of identical fp32 operations; h differs at most by the
    # last-place difference between libm's expf and a correctly rounded exp, and z inherits it
    np.testing.assert_allclose(h, hh, rtol=4 * U32, atol=4 * U32 * np.abs(hh).max())
    np.testing.assert_allclose(z, zz, rtol=0, atol=16 * U32 * np.abs(zz).max())


def test_ffn_f32_within_the_fp32_bound_of_the_fp64_statement():
    """At the tiny workload's shape: |z32 - z64| stays inside a first-order bound of fp32
    sequential summation (gamma_n = n u / (1 - n u) times the sums of absolute terms),
    propagated through SwiGLU, with a factor 2 for the second-order terms."""
    d, f = 512, 256
    for e in (0, 5):
        ex = syn.expert_tensors(0, 0, e, d, f, -8, -4)
        x = syn.activations(0, 0, 1, d)[0]
        h32, z32 = oracle.expert_ffn_f32(x, ex)
        h64, z64 = oracle.expert_ffn(x, ex)
        xv = bf16_to_f64(x)
        Wg, Wu, Wd = (decode_matrix(ex[m + "_q"], ex[m + "_s"]) for m in ("gate", "up", "down"))
        gam = lambda n: n * U32 / (1 - n * U32)
        g, u = Wg @ xv, Wu @ xv
        dg, du = gam(d) * (np.abs(Wg) @ np.abs(xv)), gam(d) * (np.abs(Wu) @ np.abs(xv))
        sig = 1 / (1 + np.exp(-g))
        dsilu = np.abs(sig * (1 + g * (1 - sig)))           # |silu'(g)|
        dh = dsilu * dg * np.abs(u) + np.abs(g * sig) * du + 6 * U32 * np.abs(h64)
        dz = np.abs(Wd) @ dh + gam(f + 1) * (np.abs(Wd) @ np.abs(h64))
        assert np.all(np.abs(h32 - h64) <= 2 * dh), np.max(np.abs(h32 - h64) / dh)
        assert np.all(np.abs(z32 - z64) <= 2 * dz), np.max(np.abs(z32 - z64) / dz)


def test_combine_f32_one_hot_and_ascending_order():
    rng = np.random.default_rng(18)
    z = rng.normal(size=(3, 16)).astype(np.float32)
    y = oracle.combine_f32(z, np.array([0.0, 1.0, 0.0], np.float32))
    np.testing.assert_array_equal(y, z[1])
    # order decides the value: in fp32, (1 + 2^24) - 2^24 = 0 (ascending j) while
    # 1 + (2^24 - 2^24) = 1 (any order that pairs the large terms first)
    z = np.array([[1.0], [2.0 ** 24], [-(2.0 ** 24)]], np.float32)
    assert oracle.combine_f32(z, np.ones(3, np.float32))[0] == 0.0
    z = np.array([[2.0 ** 24], [-(2.0 ** 24)], [1.0]], np.float32)
    assert oracle.combine_f32(z, np.ones(3, np.float32))[0] == 1.0


# ----------------------------------------------------------------------------- layer

def _tiny_layer_inputs(seed=0):
    """The tiny configuration: d=512, f=256, E=16, k=2, T=4, identity slots, seed 0."""
    d, f, E, k, T = 512, 256, 16, 2, 4
    x = syn.activations(seed, 0, T, d)
    wr = syn.router_weight(seed, 0, E, d)
    tab = syn.identity_slot_table(E)
    experts = [syn.expert_tensors(seed, 0, e, d, f, -8, -4) for e in range(E)]
    stacked = {n: np.stack([ex[n] for ex in experts]) for n in syn.EXPERT_TENSORS}
    return d, f, E, k, T, x, wr, tab, experts, stacked


def test_tiny_layer_against_independent_rederivation():
    d, f, E, k, T, x, wr, tab, experts, stacked = _tiny_layer_inputs()
    r = oracle.moe_layer(x, wr, None, tab, k, stacked, precision="f64")
    r32 = oracle.moe_layer(x, wr, None, tab, k, stacked)       # the fp32 reference statement
    assert r["status"] == 0 and r32["status"] == 0
    np.testing.assert_array_equal(r32["ids"], r["ids"])
    np.testing.assert_array_equal(r32["weights"], r["weights"])
    for t in range(T):
        keys, s32 = [], {}
        for e in range(E):
            ex = sum((bf16_exact(int(a)) * bf16_exact(int(b)) for a, b in zip(x[t], wr[e])), Fraction(0))
            l32 = round_fraction_to_f32(ex)
            s32[e] = np.float32(1.0 / (1.0 + math.exp(-float(l32))))
            keys.append((-float(s32[e]), e))
        chosen = sorted(e for _, e in sorted(keys)[:k])
        assert r["ids"][t].tolist() == chosen
        tot = np.float32(0)
        for e in chosen:
            tot = np.float32(tot + s32[e])
        xv = bf16_to_f64(x[t])
        y = np.zeros(d)
        for e in chosen:
            ex = experts[tab[e]]
            g = decode_matrix(ex["gate_q"], ex["gate_s"]) @ xv
            u = decode_matrix(ex["up_q"], ex["up_s"]) @ xv
            hh = g * u / (1 + np.exp(-g))
            y += float(np.float32(s32[e] / tot)) * (decode_matrix(ex["down_q"], ex["down_s"]) @ hh)
        np.testing.assert_allclose(r["y"][t], y, rtol=1e-9, atol=1e-9 * np.abs(y).max())
        assert np.abs(r32["y"][t] - y).max() <= 1e-5 * np.abs(y).max()
        # bf16 output is the one-step rounding of y
        yb = syn.bf16_bits_to_f32(r["y_bf16"][t]).astype(np.float64)
        assert np.all(np.abs(yb - r["y"][t]) <= np.abs(r["y"][t]) * 2.0 ** -8 + 1e-300)


def test_layer_invariant_under_slot_relabelling_and_token_order():
    d, f, E, k, T, x, wr, tab, experts, stacked = _tiny_layer_inputs(seed=3)
    base = oracle.moe_layer(x, wr, None, tab, k, stacked)
    perm = np.random.default_rng(9).permutation(E)          # expert e now lives in slot perm[e]
    tab2 = perm.astype(np.int32)
    stacked2 = {n: np.empty_like(a) for n, a in stacked.items()}
    for e in range(E):
        for n in stacked:
            stacked2[n][perm[e]] = stacked[n][e]
    r2 = oracle.moe_layer(x, wr, None, tab2, k, stacked2)
    np.testing.assert_array_equal(r2["y"], base["y"])
    np.testing.assert_array_equal(r2["ids"], base["ids"])
    order = np.array([2, 0, 3, 1])
    r3 = oracle.moe_layer(x[order], wr, None, tab, k, stacked)
    np.testing.assert_array_equal(r3["y"], base["y"][order])


def test_residual_rmsnorm_against_numpy():
    rng = np.random.default_rng(10)
    T, d = 3, 256
    x = syn.f32_to_bf16_bits(rng.normal(size=(T, d)).astype(np.float32))
    y = rng.normal(size=(T, d)) * 0.3
    out = oracle.residual_rmsnorm(x, y, 1e-6)
    v = bf16_to_f64(x) + y
    ref = v / np.sqrt(np.mean(v * v, axis=1, keepdims=True) + 1e-6)
    got = syn.bf16_bits_to_f32(out).astype(np.float64)
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)


def test_expert_size_matches_the_pages():
    g = dict(l.split() for l in open(os.path.join(GOLDEN, "expert_bytes.txt")) if l.strip() and not l.startswith("#"))
    d, f = int(g["d"]), int(g["f"])
    b = oracle.expert_bytes(d, f)
    assert b == 18_800_640
    assert round(b / 1e6, 1) == float(g["bytes_per_expert_mb"])
    n = int(g["experts_total"])
    assert round(n * b / 1e9, 1) == float(g["bytes_total_gb"])
    assert round(n * 3 * d * f / 1e9, 1) == float(g["weights_total_billion"])


# ----------------------------------------------------------------- cache-conditional routing

def test_residency_bias_hand_worked():
    """Hand values: slots 0..3 hold experts 4, 1, -, 2, so experts 1, 2 and 4 are resident;
    expert 0 maps to slot 3 (which holds 2), expert 3 has no slot, expert 5 points outside the
    slot range."""
    tab = np.array([3, 1, 3, -1, 0, 7], np.int32)
    res = np.array([4, 1, -1, 2], np.int32)
    bias = np.array([0.25, -0.5, 0.125, 1.0, 1.0, 0.0], np.float32)
    got = oracle.residency_bias(bias, tab, res, 0.5)
    assert got.tolist() == [0.25, 0.0, 0.625, 1.0, 1.5, 0.0]
    # one fp32 rounding: 1 + 2^-25 rounds back to 1, 1 + 3*2^-24 rounds to 1 + 2^-22
    got = oracle.residency_bias(bias, tab, res, 2.0 ** -25)
    assert got[4] == np.float32(1.0) and got[1] == np.float32(-0.5 + 2.0 ** -25)
    got = oracle.residency_bias(bias, tab, res, 3 * 2.0 ** -24)
    assert got[4] == np.float32(1.0 + 2.0 ** -22)
    assert oracle.residency_bias(None, tab, res, 0.5).tolist() == [0.0, 0.5, 0.5, 0.0, 0.5, 0.0]


def _brute_route(x, wr, bias, k):
    """Top-k by python sort of (-(s + bias) in fp32, id) over every expert, weights s / sum."""
    T, E = x.shape[0], wr.shape[0]
    ids, ws = [], []
    for t in range(T):
        s = [np.float32(1.0 / (1.0 + math.exp(-float(round_fraction_to_f32(
            sum((bf16_exact(int(a)) * bf16_exact(int(b)) for a, b in zip(x[t], wr[e])), Fraction(0)))))))
            for e in range(E)]
        keys = sorted((-float(np.float32(s[e] + bias[e])), e) for e in range(E))
        chosen = sorted(e for _, e in keys[:k])
        tot = np.float32(0)
        for e in chosen:
            tot = np.float32(tot + s[e])
        ids.append(chosen)
        ws.append([np.float32(s[e] / tot) for e in chosen])
    return np.array(ids, np.int32), np.array(ws, np.float32)


def test_cache_conditional_routing_limits():
    """Soft residency bias on tiny random routers: it never masks (every expert keeps its slot),
    lambda = 0 is the exact routing, a large lambda picks only resident experts (the hard mask's
    choice when the masked keys are separated), and a moderate lambda still lets a strong
    non-resident expert through; every case matches a brute-force restatement."""
    rng = np.random.default_rng(12)
    T, d, E, k = 4, 64, 12, 3
    saw_nonresident = 0
    for trial in range(12):
        x = syn.f32_to_bf16_bits(rng.normal(size=(T, d)).astype(np.float32))
        wr = syn.f32_to_bf16_bits((rng.normal(size=(E, d)) * 0.08).astype(np.float32))
        tab = rng.permutation(E).astype(np.int32)
        res = np.full(E, -1, np.int32)
        on = rng.choice(E, 5, replace=False)
        res[tab[on]] = on
        bias = (rng.normal(size=E) * 0.02).astype(np.float32) if trial % 2 else None
        b0 = np.zeros(E, np.float32) if bias is None else bias
        exact = oracle.route_topk(x, wr, bias, tab, k)
        for lam in (0.0, 0.03, 1.0):
            rb = oracle.residency_bias(bias, tab, res, lam)
            r = oracle.route_topk(x, wr, rb, tab, k)
            assert r["status"] == 0
            ids, ws = _brute_route(x, wr, rb, k)
            np.testing.assert_array_equal(r["ids"], ids)
            np.testing.assert_array_equal(r["weights"], ws)
            np.testing.assert_array_equal(r["slots"], tab[r["ids"]])
            if lam == 0.0:
                np.testing.assert_array_equal(r["ids"], exact["ids"])
                np.testing.assert_array_equal(r["weights"], exact["weights"])
            if lam == 1.0:
                assert np.isin(r["ids"], on).all()
                masked_tab = np.where(np.isin(np.arange(E), on), tab, -1).astype(np.int32)
                m = oracle.route_topk(x, wr, bias, masked_tab, k, want_logits=True)
                for t in range(T):
                    kv = np.sort((m["scores"][t] + b0)[on])[::-1]
                    if kv[k - 1] - kv[k] > 2.0 ** -20:
                        np.testing.assert_array_equal(r["ids"][t], m["ids"][t])
                        np.testing.assert_array_equal(r["weights"][t], m["weights"][t])
            if lam == 0.03:
                saw_nonresident += int((~np.isin(r["ids"], on)).sum())
    assert saw_nonresident > 0


# ----------------------------------------------------------------------------- cb3 codec

E2M1_CODE = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}


def _fp4_row(values, scale_bytes):
    """Pack K values (each an e2m1 value times its block's 2^(b-127)) into codes + scales."""
    K = len(values)
    q = np.zeros(K // 2, np.uint8)
    for k, v in enumerate(values):
        m = abs(v) / 2.0 ** (int(scale_bytes[k // 32]) - 127)
        c = E2M1_CODE[m] | (8 if v < 0 else 0)
        q[k // 2] |= c << (4 * (k % 2))
    return q, np.asarray(scale_bytes, np.uint8)


def _levels(cb):
    return [oracle.bf16_value(int(b)) for b in cb]


SIGNED_E2M1 = [0.0] + [sg * m for m in (0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0) for sg in (1.0, -1.0)]


def test_cb3_lossless_rows():
    """A row with at most 8 distinct values is reproduced exactly: its levels are those values,
    ascending, then zeros."""
    rng = np.random.default_rng(31)
    for trial in range(20):
        nv = int(rng.integers(1, 9))
        vals = [float(v) for v in rng.choice(SIGNED_E2M1, nv, replace=False)]
        b = int(rng.integers(100, 140))
        row = [v * 2.0 ** (b - 127) for v in rng.choice(vals, 64)]
        q, s = _fp4_row(row, [b, b])
        cb, idx, n = oracle.cb3_pack_row(q, s)
        distinct = sorted(set(row))
        assert n == len(distinct)
        lv = _levels(cb)
        assert lv[:n] == distinct and all(v == 0.0 for v in lv[n:])
        assert [lv[i] for i in idx] == row


def test_cb3_equal_cost_tie_goes_to_the_earlier_split():
    """Nine equally spaced values (-4..4), 32 of each: every merge of two neighbours costs the
    same (16); the smallest split point on ties merges the top pair, 3 and 4 -> 3.5."""
    vals = [-4.0, -3.0, -2.0, -1.0, 0.0, 1.0, 2.0, 3.0, 4.0]
    row = [v for v in vals for _ in range(32)]
    q, s = _fp4_row(row, [127] * 9)
    cb, idx, n = oracle.cb3_pack_row(q, s)
    assert n == 9
    assert _levels(cb) == [-4.0, -3.0, -2.0, -1.0, 0.0, 1.0, 2.0, 3.5]
    assert idx.tolist() == [min(i // 32, 7) for i in range(288)]


def _set_partitions(n, blocks):
    """Every partition of range(n) into exactly `blocks` non-empty sets (restricted growth)."""
    a = [0] * n

    def rec(i, m):
        if i == n:
            if m == blocks:
                yield list(a)
            return
        if blocks - m > n - i:
            return
        for v in range(min(m + 1, blocks)):
            a[i] = v
            yield from rec(i + 1, max(m, v + 1))

    yield from rec(0, 0)


def test_cb3_optimal_among_all_partitions():
    """Rows with 9 or 10 distinct values and uneven counts: the oracle's clusters reach the
    least squared error over every partition of the distinct values into 8 sets (not only
    contiguous ones), computed in exact rationals; each level is bf16 of its cluster's exact
    mean and the levels ascend."""
    rng = np.random.default_rng(32)
    for trial in range(8):
        nd = 9 + trial % 2
        vals = [float(v) for v in rng.choice(SIGNED_E2M1, nd, replace=False)]
        row = vals + [float(v) for v in rng.choice(vals, 64 - nd, p=rng.dirichlet(np.ones(nd)))]
        rng.shuffle(row)
        q, s = _fp4_row(row, [127, 127])
        cb, idx, n = oracle.cb3_pack_row(q, s)
        u = sorted(set(row))
        assert n == len(u) == nd
        cnt = {v: row.count(v) for v in u}

        def sse(groups):
            tot = Fraction(0)
            for g in groups:
                c = sum(cnt[v] for v in g)
                mean = sum(Fraction(v) * cnt[v] for v in g) / c
                tot += sum(cnt[v] * (Fraction(v) - mean) ** 2 for v in g)
            return tot

        best = min(sse([[u[i] for i in range(n) if p[i] == b] for b in range(8)]) for p in _set_partitions(n, 8))
        got_groups = [sorted({row[k] for k in range(64) if idx[k] == g}) for g in range(8)]
        assert all(got_groups), got_groups
        assert sum(len(g) for g in got_groups) == n         # every value in exactly one cluster
        assert sse(got_groups) == best
        lv = _levels(cb)
        assert lv == sorted(lv)
        for g, grp in enumerate(got_groups):
            mean = sum(Fraction(v) * cnt[v] for v in grp) / sum(cnt[v] for v in grp)
            assert lv[g] == round_fraction_to_bf16(mean), (g, grp)


def round_fraction_to_bf16(v: Fraction) -> float:
    """Nearest bf16 to an exact rational, ties to even (normal range)."""
    if v == 0:
        return 0.0
    sgn = -1 if v < 0 else 1
    a = abs(v)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (e - 7)
    r = a / quantum
    fl = math.floor(r)
    rem = r - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sgn * float(fl * quantum)


def test_cb3_ffn_equals_fp4_ffn_on_lossless_expert():
    """An expert whose rows hold at most 8 distinct values packs losslessly, so the cb3 FFN
    equals the FP4 FFN exactly (same products, same order)."""
    rng = np.random.default_rng(33)
    d, f = 64, 32
    ex = {}
    for m, (R, K) in (("gate", (f, d)), ("up", (f, d)), ("down", (d, f))):
        qs, ss = [], []
        for r in range(R):
            b = int(rng.integers(122, 128))
            mags = rng.choice([0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], 4, replace=False)
            vals = [float(v) * 2.0 ** (b - 127) for v in np.concatenate([mags, -mags])]
            q, s = _fp4_row([float(v) for v in rng.choice(vals, K)], [b] * (K // 32))
            qs.append(q)
            ss.append(s)
        ex[m + "_q"], ex[m + "_s"] = np.stack(qs), np.stack(ss)
    cx = oracle.cb3_pack_expert(ex)
    for t in range(3):
        x = syn.f32_to_bf16_bits(rng.normal(size=d).astype(np.float32))
        h1, z1 = oracle.expert_ffn(x, ex)
        h2, z2 = oracle.cb3_expert_ffn(x, cx)
        np.testing.assert_array_equal(h1, h2)
        np.testing.assert_array_equal(z1, z2)
