"""Pins for the oracle's quantizer (a1) against hand-worked fixtures, the
error bound, exact rational re-encoding and per-group closed forms.
Source: TailorKV article §2.2 (quant_1bit snippet); on-device article §3.1."""
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import kvq_oracle as O

pytestmark = pytest.mark.cpu


def _load_quant_cases(golden_dir):
    cases = []
    with open(os.path.join(golden_dir, "quant_rounding.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            b, xs, codes, scale, zero = [c.strip() for c in line.split("|")]
            cases.append((int(b), [float(v) for v in xs.split()],
                          [int(v) for v in codes.split()], float(scale), float(zero)))
    return cases


def test_golden_rounding(golden_dir):
    cases = _load_quant_cases(golden_dir)
    assert len(cases) >= 6
    for b, xs, codes, scale, zero in cases:
        c, s16, z16, s32 = O.quantize_groups(np.array([xs], dtype=np.float16), b)
        assert c[0].tolist() == codes, (b, xs)
        assert float(s16[0]) == scale and float(z16[0]) == zero


def test_golden_third_scale(golden_dir):
    # 2-bit group [0, .25, .5, 1]: scale = fl32(1/3); quotients 0.75, 1.5, 3 after
    # fp32 rounding -> codes 0,1,2,3 (1.5 rounds to even 2).
    c, s16, z16, s32 = O.quantize_groups(np.array([[0.0, 0.25, 0.5, 1.0]], np.float16), 2)
    assert c[0].tolist() == [0, 1, 2, 3]
    assert s32[0] == np.float32(1.0) / np.float32(3.0)
    assert s16[0] == np.float16(s32[0])


@pytest.mark.parametrize("bits", [1, 2, 4, 8])
def test_error_bound_and_range(bits):
    rng = np.random.default_rng(100 + bits)
    x = (rng.standard_normal((500, 64)) * rng.choice([1.0, 10.0], size=(500, 1))).astype(np.float16)
    codes, s16, z16, s32 = O.quantize_groups(x, bits)
    L = 2 ** bits - 1
    assert codes.min() >= 0 and codes.max() <= L
    xf = x.astype(np.float64)
    mn = xf.min(axis=1)
    mx = xf.max(axis=1)
    # code(min) = 0 and code(max) = 2^b - 1
    assert np.all(codes[np.arange(500), xf.argmin(axis=1)] == 0)
    assert np.all(codes[np.arange(500), xf.argmax(axis=1)] == L)
    # |x - (min + code*scale32)| <= scale32 * (1/2 + (2^b-1) 2^-23), in fp64: the
    # fp32 quotient u <= 2^b-1 carries one rounding of at most u 2^-24.
    slack = 0.5 + L * 2.0 ** -23
    rec = mn[:, None] + codes * s32.astype(np.float64)[:, None]
    err = np.abs(xf - rec)
    assert np.all(err <= s32.astype(np.float64)[:, None] * slack)
    assert np.max(err / s32.astype(np.float64)[:, None]) > 0.49   # the bound is tight
    # with the stored fp16 scale: add (2^b-1) |scale32 - scale16|
    rec16 = z16.astype(np.float64)[:, None] + codes * s16.astype(np.float64)[:, None]
    bound = s32.astype(np.float64) * slack + L * np.abs(
        s32.astype(np.float64) - s16.astype(np.float64))
    assert np.all(np.abs(xf - rec16) <= bound[:, None] + 1e-12)
    assert np.array_equal(z16.astype(np.float64), mn)


@pytest.mark.parametrize("bits", [1, 2, 4, 8])
def test_exact_rational_reencode(bits):
    """Exact rational arithmetic (no fp rounding) gives the same codes except
    where the exact quotient lies within 1e-6 of a half-integer."""
    rng = np.random.default_rng(7 + bits)
    x = rng.standard_normal((40, 64)).astype(np.float16)
    codes, _, _, _ = O.quantize_groups(x, bits)
    L = 2 ** bits - 1
    mism = 0
    for r in range(x.shape[0]):
        vals = [Fraction(float(v)) for v in x[r]]
        mn, mx = min(vals), max(vals)
        for i, v in enumerate(vals):
            u = (v - mn) * L / (mx - mn)
            fl = u.numerator // u.denominator
            frac = u - fl
            if frac > Fraction(1, 2) or (frac == Fraction(1, 2) and fl % 2 == 1):
                fl += 1
            want = min(max(fl, 0), L)
            if abs(frac - Fraction(1, 2)) < Fraction(1, 10 ** 6):
                continue
            mism += int(want != codes[r, i])
    assert mism == 0


def test_one_bit_is_midpoint_threshold():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((300, 64)).astype(np.float16)
    codes, _, _, _ = O.quantize_groups(x, 1)
    xf = x.astype(np.float64)
    mn = xf.min(axis=1, keepdims=True)
    mx = xf.max(axis=1, keepdims=True)
    mid = (mx - mn) / 2
    rel = (xf - mn) - mid
    clear = np.abs(rel) > 1e-6 * (mx - mn)
    assert np.array_equal(codes[clear], (rel > 0)[clear].astype(np.int64))


@pytest.mark.parametrize("bits", [1, 2, 4, 8])
def test_k_grouping_per_channel_64_tokens(bits):
    """Group (g, c) of K holds tokens 64g..64g+63 of channel c: build K so every
    group spans a known interval [lo, hi] and check the stored zero/scale."""
    T, d = 64 * 3 + 10, 6
    rng = np.random.default_rng(11)
    lo = np.round(rng.uniform(-8, 0, size=(3, d)) * 4) / 4
    hi = lo + np.round(rng.uniform(1, 8, size=(3, d)) * 4) / 4
    K = np.zeros((T, d))
    for g in range(3):
        for c in range(d):
            vals = rng.uniform(lo[g, c], hi[g, c], size=64)
            vals[5] = lo[g, c]
            vals[40] = hi[g, c]
            K[64 * g:64 * g + 64, c] = vals
    K[192:] = rng.standard_normal((10, d))
    K16 = K.astype(np.float16)
    pk = O.pack_k(K16, bits)
    assert pk["n_packed"] == 192
    L = 2 ** bits - 1
    for g in range(3):
        for c in range(d):
            assert float(pk["zero16"][g, c]) == float(np.float16(lo[g, c]))
            s = (np.float32(np.float16(hi[g, c])) - np.float32(np.float16(lo[g, c]))) / np.float32(L)
            assert pk["scale32"][g, c] == s
            assert pk["codes"][64 * g + 5, c] == 0 and pk["codes"][64 * g + 40, c] == L
    assert np.array_equal(pk["tail"], K16[192:])
    dq = O.dequant_k(pk)
    assert np.array_equal(dq[192:], K16[192:].astype(np.float64))


@pytest.mark.parametrize("gd", [32, 64])
def test_v_grouping_per_token(gd):
    T, d = 5, 128
    rng = np.random.default_rng(5)
    V = rng.standard_normal((T, d)).astype(np.float16)
    pv = O.pack_v(V, 4, gd)
    assert pv["zero16"].shape == (T, d // gd)
    for t in range(T):
        for j in range(d // gd):
            seg = V[t, j * gd:(j + 1) * gd].astype(np.float32)
            assert pv["zero16"][t, j] == np.float16(seg.min())
            assert pv["scale32"][t, j] == (seg.max() - seg.min()) / np.float32(15)


def test_sixteen_bit_is_nearly_lossless():
    """At b=16 the only loss left is the fp16 rounding of the stored scale:
    |x - x_hat| <= range * 2^-11 (+ the half-step range/65535/2)."""
    rng = np.random.default_rng(9)
    V = (rng.standard_normal((64, 128)) * 3).astype(np.float16)
    pv = O.pack_v(V, 16, 64)
    err = np.abs(O.dequant_v(pv) - V.astype(np.float64))
    rng_g = np.ptp(V.astype(np.float64).reshape(64, 2, 64), axis=2).repeat(64, axis=1)
    assert np.all(err <= rng_g * (2.0 ** -11 + 0.5 / 65535))


# ---- symmetric V quantization   [on-device article §3.1: V INT4 symmetric, group quantization]

def test_golden_symmetric_groups(golden_dir):
    import os
    n = 0
    with open(os.path.join(golden_dir, "sym_v_small.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            bits, xs, cs, sc = [c.strip() for c in line.split("|")]
            x = np.array([float(v) for v in xs.split()], np.float16)
            codes, s16, s32 = O.quantize_groups_sym(x, int(bits))
            assert codes.tolist() == [int(v) for v in cs.split()]
            assert float(s32) == float(sc) and float(s16) == float(sc)
            n += 1
    assert n == 4


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_symmetric_bound_range_and_extremes(bits):
    """|x - code * scale32| <= scale32 / 2 (fp64, plus the one-rounding slack L * 2^-23 of the
    fp32 quotient), codes in [-L, L], max |x| -> +-L."""
    rng = np.random.default_rng(60 + bits)
    x = (rng.standard_normal((500, 64)) * rng.choice([0.01, 1, 30], size=(500, 1))).astype(np.float16)
    codes, s16, s32 = O.quantize_groups_sym(x, bits)
    L = 2 ** (bits - 1) - 1
    assert codes.min() >= -L and codes.max() <= L
    err = np.abs(x.astype(np.float64) - codes * s32.astype(np.float64)[:, None])
    assert np.all(err <= s32.astype(np.float64)[:, None] * (0.5 + L * 2.0 ** -23))
    i = np.argmax(np.abs(x.astype(np.float32)), axis=1)
    assert np.all(np.abs(codes[np.arange(500), i]) == L)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_symmetric_mirror(bits):
    """A group and its negation get the same scale and negated codes (ties go to even either way)."""
    rng = np.random.default_rng(70 + bits)
    x = rng.standard_normal((300, 32)).astype(np.float16)
    c1, s1, _ = O.quantize_groups_sym(x, bits)
    c2, s2, _ = O.quantize_groups_sym(-x, bits)
    assert np.array_equal(c1, -c2) and np.array_equal(s1.view(np.uint16), s2.view(np.uint16))


def test_symmetric_exact_rounding_away_from_ties():
    """Codes equal the exact rational round-to-nearest of x / scale32 where the quotient is not
    within 1e-6 of a half-integer (computed with Python fractions)."""
    from fractions import Fraction
    rng = np.random.default_rng(80)
    x = rng.standard_normal((200, 16)).astype(np.float16)
    codes, _, s32 = O.quantize_groups_sym(x, 4)
    for g in range(200):
        sc = Fraction(float(s32[g]))
        for k in range(16):
            q = Fraction(float(x[g, k])) / sc
            frac = q - (q.numerator // q.denominator)
            if abs(frac - Fraction(1, 2)) < Fraction(1, 10 ** 6):
                continue
            want = max(-7, min(7, round(q)))
            assert codes[g, k] == want


def test_symmetric_dequant_and_attention():
    """The symmetric cache dequantizes to code * scale16; attention over it stays close to
    attention over the fp16 values (4-bit, G 32)."""
    rng = np.random.default_rng(81)
    V = rng.standard_normal((400, 128)).astype(np.float16)
    pv = O.pack_v_sym(V, 4, 32)
    vh = O.dequant_v(pv)
    j = np.arange(128) // 32
    assert np.array_equal(vh, pv["codes"] * pv["scale16"].astype(np.float64)[:, j])
    assert np.max(np.abs(vh - V.astype(np.float64))) <= np.max(pv["scale32"]) * 0.51 + 1e-3


# ---- outlier-channel isolation   [meeting article §8.2]

def test_outlier_channels_find_planted_channels_and_break_ties_low():
    rng = np.random.default_rng(90)
    K = rng.standard_normal((1000, 128)).astype(np.float32)
    K[:, [7, 70, 99]] *= [10, 20, 5]
    K = K.astype(np.float16)
    assert O.outlier_channels(K, 1).tolist() == [70]
    assert O.outlier_channels(K, 3).tolist() == [7, 70, 99]
    # identical channels: the lower one first
    K2 = np.zeros((64, 128), np.float16)
    K2[::2, 3] = 1
    K2[::2, 9] = 1
    assert O.outlier_channels(K2, 1).tolist() == [3]


def test_outlier_variance_brute_force():
    """Small integer keys: the chosen channels are the n largest exact variances (fractions), ties
    low -- except where two exact variances at the boundary lie within fp64 rounding of each
    other (1e-12 relative), where the fp64 definition may order them either way."""
    from fractions import Fraction
    rng = np.random.default_rng(91)
    for _ in range(10):
        T, d, n = int(rng.integers(2, 40)), 16, int(rng.integers(1, 5))
        K = rng.integers(-4, 5, size=(T, d)).astype(np.float16)
        var = []
        for c in range(d):
            xs = [Fraction(int(x)) for x in K[:, c]]
            m = sum(xs) / T
            var.append(sum((x - m) ** 2 for x in xs) / T)
        want = sorted(sorted(range(d), key=lambda c: (-var[c], c))[:n])
        got = O.outlier_channels(K, n).tolist()
        for a in set(got) ^ set(want):          # exchanged at the boundary: near-equal variances only
            b = sorted(range(d), key=lambda c: (-var[c], c))[n - 1 if a not in want else n]
            assert abs(float(var[a]) - float(var[b])) <= 1e-12 * max(1.0, abs(float(var[b]))), (got, want)


def test_channel_variance_exact_sums_order_independent_and_near_exact():
    """The sums are exact, so any token order gives the same bits (a plain fp64 running sum of
    these squares does not: values near 2^-14 and near 2^8 need more than 53 bits together); and
    the result lies within a few roundings of the exact (fraction) variance, mean of the order of
    the spread here so the subtraction does not cancel."""
    from fractions import Fraction
    rng = np.random.default_rng(94)
    T = 3000
    K = (rng.standard_normal((T, 8)) * np.array([1e-4, 1e-3, 1, 30, 200, 1, 5e-4, 2])).astype(np.float16)
    K[::7, 0] = np.float16(300.0)                  # tiny and large values in one channel
    v = O.channel_variance(K)
    perm = rng.permutation(T)
    assert np.array_equal(O.channel_variance(K[perm]).view(np.uint64), v.view(np.uint64))
    assert np.array_equal(O.channel_variance(K[::-1]).view(np.uint64), v.view(np.uint64))
    for c in range(8):
        xs = [Fraction(float(x)) for x in K[:, c]]
        m = sum(xs) / T
        exact = sum((x - m) ** 2 for x in xs) / T
        assert abs(v[c] - float(exact)) <= 1e-13 * float(exact), c
    # constant channel: zero variance; a single token: zero
    Kc = np.full((100, 4), np.float16(3.5))
    assert np.all(O.channel_variance(Kc) == 0.0)
    assert np.all(O.channel_variance(K[:1]) == 0.0)


def test_pack_k_outlier_keeps_outliers_exact_and_the_rest_unchanged():
    rng = np.random.default_rng(92)
    K = (rng.standard_normal((64 * 5 + 9, 128)) * np.where(rng.random(128) < 0.05, 10, 1)).astype(np.float16)
    ch = O.outlier_channels(K, 4)
    po, pk = O.pack_k_outlier(K, 4, ch), O.pack_k(K, 4)
    normal = np.setdiff1d(np.arange(128), ch)
    assert np.array_equal(po["codes"][:, normal], pk["codes"][:, normal])
    assert np.array_equal(po["scale16"][:, normal].view(np.uint16), pk["scale16"][:, normal].view(np.uint16))
    dq, dk = O.dequant_k(po), O.dequant_k(pk)
    assert np.array_equal(dq[:, ch], K[:, ch].astype(np.float64))          # outliers exact (packed and tail)
    assert np.array_equal(dq[:, normal], dk[:, normal])
    assert np.all(po["codes"][:, ch] == 0) and np.all(po["scale16"][:, ch] == 0)
    # no outliers: the plain pack
    pe = O.pack_k_outlier(K, 4, [])
    assert np.array_equal(O.dequant_k(pe), dk)


def test_all_channels_outliers_is_attention_over_fp16_keys():
    rng = np.random.default_rng(93)
    K = rng.standard_normal((200, 128)).astype(np.float16)
    V = rng.standard_normal((200, 128)).astype(np.float16)
    q = rng.standard_normal(128).astype(np.float16)
    po = O.pack_k_outlier(K, 1, np.arange(128))
    pv = O.pack_v(V, 1, 64)
    o = O.decode_attn_quant(q[None], [po], [pv])[0]
    ref, _ = O.softmax_attention(q, K, O.dequant_v(pv))
    assert np.allclose(o, ref, rtol=0, atol=1e-12)
