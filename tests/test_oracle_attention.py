"""Pins for the oracle's attention paths (a3 quantized decode, a6 sparse
attention) against an independently written brute-force two-pass softmax,
closed forms and the b=16 / full-selection reductions.
Sources: on-device article §3.2; meeting article §3.2; TailorKV §2.2-2.3."""
import math

import numpy as np
import pytest

from oracle import kvq_oracle as O

pytestmark = pytest.mark.cpu


def brute_attention(q, K, V):
    """Two explicit passes with Python floats: max, then exp-sum and weighted sum."""
    d = len(q)
    s = [sum(float(q[c]) * float(K[t][c]) for c in range(d)) / math.sqrt(d) for t in range(len(K))]
    m = max(s)
    w = [math.exp(x - m) for x in s]
    z = sum(w)
    return [sum(w[t] * float(V[t][c]) for t in range(len(K))) / z for c in range(len(V[0]))]


@pytest.mark.parametrize("T,d", [(1, 4), (7, 4), (16, 8), (33, 16)])
def test_softmax_attention_vs_brute_force(T, d):
    rng = np.random.default_rng(T * 100 + d)
    q = rng.standard_normal(d) * 2
    K = rng.standard_normal((T, d))
    V = rng.standard_normal((T, d))
    o, p = O.softmax_attention(q, K, V)
    ref = brute_attention(q, K, V)
    assert np.allclose(o, ref, rtol=0, atol=1e-12)
    assert abs(p.sum() - 1) < 1e-12


def test_closed_forms():
    rng = np.random.default_rng(1)
    V = rng.standard_normal((10, 4))
    K = np.tile(rng.standard_normal(4), (10, 1))       # equal keys -> uniform
    o, p = O.softmax_attention(rng.standard_normal(4), K, V)
    assert np.allclose(o, V.mean(axis=0), atol=1e-14)
    o, _ = O.softmax_attention(np.zeros(4), rng.standard_normal((10, 4)), V)
    assert np.allclose(o, V.mean(axis=0), atol=1e-14)
    # two keys: p0 = 1 / (1 + exp(s1 - s0))
    q = np.array([1.0, 0, 0, 0])
    K = np.array([[2.0, 0, 0, 0], [0.0, 0, 0, 0]])
    _, p = O.softmax_attention(q, K, V[:2])
    assert abs(p[0] - 1 / (1 + math.exp(-2.0 / 2.0))) < 1e-15


def _cache(T, d, Hkv, seed, outliers=True):
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((Hkv, T, d))
    if outliers:
        K[:, :, [3, 17, 64, 101]] *= 10
    V = rng.standard_normal((Hkv, T, d))
    return K.astype(np.float16), V.astype(np.float16)


@pytest.mark.parametrize("T,bits", [(64, 16), (100, 16), (257, 16), (257, 8), (130, 4), (200, 1)])
def test_quant_attention_within_perturbation_bound(T, bits):
    """Quantized decode attention vs dense fp16 attention obeys the bound that
    follows from the dequantization error alone: with ds = max_t sum_c
    |q_c| |k_hat - k| / sqrt(d) and dv = max |v_hat - v|, every probability
    moves by a factor within exp(+-2 ds), so |o - o_dense| <= (exp(2 ds) - 1)
    max|v| + dv.  A wrong sign, index or scale in the oracle breaks it."""
    d, Hq, Hkv = 128, 8, 2
    K, V = _cache(T, d, Hkv, T)
    q = np.random.default_rng(2).standard_normal((Hq, d)).astype(np.float16)
    pk = [O.pack_k(K[g], bits) for g in range(Hkv)]
    pv = [O.pack_v(V[g], bits, 64) for g in range(Hkv)]
    o = O.decode_attn_quant(q, pk, pv)
    for h in range(Hq):
        g = h // 4
        Kd, Vd = K[g].astype(np.float64), V[g].astype(np.float64)
        ref, _ = O.softmax_attention(q[h].astype(np.float64), Kd, Vd)
        ek = np.abs(O.dequant_k(pk[g]) - Kd)
        ds = np.max(ek @ np.abs(q[h].astype(np.float64))) / math.sqrt(d)
        vh = O.dequant_v(pv[g])
        dv = np.max(np.abs(vh - Vd))
        bound = (math.exp(2 * ds) - 1) * np.max(np.abs(vh)) + dv
        assert np.max(np.abs(o[h] - ref)) <= bound * (1 + 1e-9) + 1e-12


@pytest.mark.parametrize("T", [64, 100, 257, 1000])
def test_sixteen_bit_quant_attention_reduces_to_dense(T):
    """TailorKV §2.2 (quantization at b bits): at b=16 the quantized decode attention
    reduces to dense fp16 attention: the residual error, left by the fp16
    rounding of the stored scale, is below 2e-3 of the value range max|v|
    and at least 5x below the b=8 error.  (The output of random-data
    attention shrinks like 1/sqrt(T), so the value range is the scale.)"""
    d, Hq, Hkv = 128, 8, 2
    K, V = _cache(T, d, Hkv, T)
    q = np.random.default_rng(2).standard_normal((Hq, d)).astype(np.float16)
    err = {}
    for bits in (8, 16):
        pk = [O.pack_k(K[g], bits) for g in range(Hkv)]
        pv = [O.pack_v(V[g], bits, 64) for g in range(Hkv)]
        o = O.decode_attn_quant(q, pk, pv)
        e = 0.0
        for h in range(Hq):
            g = h // 4
            ref, _ = O.softmax_attention(q[h].astype(np.float64), K[g].astype(np.float64),
                                         V[g].astype(np.float64))
            e = max(e, np.max(np.abs(o[h] - ref)) / np.max(np.abs(V[g].astype(np.float64))))
        err[bits] = e
    assert err[16] < 2e-3
    assert err[16] * 5 < err[8]


def test_quant_attention_uses_tail_exactly_and_gqa_mapping():
    """T=70: 64 packed tokens + 6 tail tokens.  A dominant query aligned with a
    tail key must reproduce that key's dequantized V; head h reads kv head
    h // (Hq/Hkv), not h % Hkv."""
    d, Hq, Hkv, T = 128, 8, 2, 70
    K, V = _cache(T, d, Hkv, 5, outliers=False)
    q = np.zeros((Hq, d), dtype=np.float16)
    target = {0: (0, 66), 1: (0, 67), 5: (1, 68), 7: (1, 3)}
    for h, (g, t) in target.items():
        q[h] = (K[g, t].astype(np.float64) * 40).astype(np.float16)
    pk = [O.pack_k(K[g], 4) for g in range(Hkv)]
    pv = [O.pack_v(V[g], 4, 32) for g in range(Hkv)]
    assert pk[0]["n_packed"] == 64 and pk[0]["tail"].shape[0] == 6
    o = O.decode_attn_quant(q, pk, pv)
    for h, (g, t) in target.items():
        vhat = O.dequant_v(pv[g])[t]
        assert np.max(np.abs(o[h] - vhat)) < 1e-3 * np.max(np.abs(vhat)) + 1e-6, h
    # head 1 is in group 0 under floor(h*Hkv/Hq); under h % Hkv it would read kv head 1
    assert O.kv_head_of(1, 8, 2) == 0 and O.kv_head_of(4, 8, 2) == 1
    assert O.kv_head_of(5, 32, 32) == 5


def test_quant_attention_matches_brute_force_on_dequantized_cache():
    d, Hq, Hkv, T = 16, 4, 2, 80
    rng = np.random.default_rng(12)
    K = rng.standard_normal((Hkv, T, d)).astype(np.float16)
    V = rng.standard_normal((Hkv, T, d)).astype(np.float16)
    q = rng.standard_normal((Hq, d)).astype(np.float16)
    pk = [O.pack_k(K[g], 2) for g in range(Hkv)]
    pv = [O.pack_v(V[g], 2, 8) for g in range(Hkv)]
    o = O.decode_attn_quant(q, pk, pv)
    for h in range(Hq):
        g = h // 2
        # dequantize by hand with explicit loops
        Kh = []
        for t in range(T):
            row = []
            for c in range(d):
                if t < 64:
                    row.append(float(pk[g]["zero16"][t // 64, c])
                               + int(pk[g]["codes"][t, c]) * float(pk[g]["scale16"][t // 64, c]))
                else:
                    row.append(float(K[g, t, c]))
            Kh.append(row)
        Vh = [[float(pv[g]["zero16"][t, c // 8]) + int(pv[g]["codes"][t, c]) * float(pv[g]["scale16"][t, c // 8])
               for c in range(d)] for t in range(T)]
        ref = brute_attention(q[h].astype(np.float64), Kh, Vh)
        assert np.allclose(o[h], ref, atol=1e-12)


def test_sparse_attention_full_selection_is_dense():
    d, T = 128, 300
    K, V = _cache(T, d, 1, 8)
    q = np.random.default_rng(4).standard_normal(d).astype(np.float16)
    sel = O.topk_select(np.zeros(T, np.float32), T, 4, 64)     # K >= T - n_s - W
    assert np.array_equal(sel, np.arange(T))
    o, p = O.sparse_attn(q, K[0], V[0], sel)
    ref, pr = O.softmax_attention(q.astype(np.float64), K[0].astype(np.float64), V[0].astype(np.float64))
    assert np.array_equal(o, ref) and np.array_equal(p, pr)


def test_sparse_attention_brute_force_and_prob_order():
    d, T = 8, 40
    rng = np.random.default_rng(21)
    K = rng.standard_normal((T, d)).astype(np.float16)
    V = rng.standard_normal((T, d)).astype(np.float16)
    q = rng.standard_normal(d).astype(np.float16)
    ids = np.array([0, 3, 9, 10, 25, 39])
    o, p = O.sparse_attn(q, K, V, ids)
    ref = brute_attention(q.astype(np.float64), K[ids].astype(np.float64), V[ids].astype(np.float64))
    assert np.allclose(o, ref, atol=1e-12)
    s = [float(np.dot(q.astype(np.float64), K[t].astype(np.float64))) / math.sqrt(d) for t in ids]
    assert int(np.argmax(p)) == int(np.argmax(s))
