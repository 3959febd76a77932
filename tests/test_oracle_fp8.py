"""Pins for the oracle's FP8 E4M3 cache format (meeting article, section 6 item 2:
FP8 E4M3 preferred where the hardware supports it): decoding from the format's
definition at hand-checked code points, encoding of every fp16 value against an
independent nearest-value search over the 256 codes, round trips, and attention
over exactly representable values."""
import numpy as np
import pytest

from oracle import kvq_oracle as O

pytestmark = pytest.mark.cpu


def test_decode_known_codes():
    got = O.fp8_e4m3_decode(np.array([0x38, 0x7E, 0x01, 0x08, 0x07, 0x80, 0xFE, 0x40, 0x3C]))
    want = [1.0, 448.0, 2.0 ** -9, 2.0 ** -6, 7 * 2.0 ** -9, -0.0, -448.0, 2.0, 1.5]
    assert got.tolist() == want
    assert np.isnan(O.fp8_e4m3_decode(np.array([0x7F, 0xFF]))).all()
    assert np.signbit(O.fp8_e4m3_decode(np.array([0x80])))[0]


def _nearest_codes(x):
    """Independent reference for non-negative fp16 values x: search all 128 non-negative
    codes for the nearest finite value (a distance table); ties to the even code; beyond
    448 (and +inf) saturate.  NaN -> -1."""
    vals = O.fp8_e4m3_decode(np.arange(128))
    ok = ~np.isnan(vals)
    xs = np.clip(np.where(np.isnan(x), 0.0, x), 0.0, 448.0)
    d = np.abs(xs[:, None] - np.where(ok, vals, np.inf)[None, :])
    dmin = d.min(axis=1, keepdims=True)
    tie = d == dmin
    # among the nearest codes prefer an even one (the lowest even code; ties span two codes)
    even = tie & (np.arange(128)[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), tie.argmax(axis=1))
    return np.where(np.isnan(x), -1, pick)


def test_encode_every_fp16_value():
    allv = np.arange(65536, dtype=np.uint16).view(np.float16)
    codes = O.fp8_e4m3_encode(allv)
    pos = allv[:32768].astype(np.float64)                  # the non-negative patterns (+0 .. +inf, NaNs)
    want = _nearest_codes(pos)
    nan = want < 0
    assert np.all(codes[:32768][nan] == 0x7F)
    assert np.array_equal(codes[:32768][~nan], want[~nan].astype(np.uint8))
    # the negative patterns carry the sign bit
    assert np.array_equal(codes[32768:][~nan], (want[~nan] | 0x80).astype(np.uint8))


def test_round_trip_of_every_finite_code():
    c = np.array([k for k in range(256) if k not in (0x7F, 0xFF)])
    v = O.fp8_e4m3_decode(c).astype(np.float16)           # every E4M3 value is an fp16 value
    assert np.array_equal(O.fp8_e4m3_encode(v), c.astype(np.uint8))


def test_attention_over_representable_values_is_exact_attention():
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 0x7E, size=(2, 300, 128))
    codes = np.where(rng.random(codes.shape) < 0.5, codes, codes | 0x80)
    K = O.fp8_e4m3_decode(codes[0]).astype(np.float16)
    V = O.fp8_e4m3_decode(codes[1]).astype(np.float16)
    q = rng.standard_normal(128).astype(np.float16)
    o8, p8 = O.fp8_attention(q, K, V)
    o, p = O.softmax_attention(q, K, V)
    assert np.array_equal(o8, o) and np.array_equal(p8, p)
