"""Pins for the oracle's H2O accumulate/evict (a7) and dense-preference score
(a8): a hand-worked fixture, an independent dict-based brute force over
several steps, conservation of probability mass, the no-eviction reduction,
the closed form for uniform attention and the 0 <= P <= n_q bound.
Sources: KV-cache survey §三.1-三.2; TailorKV §2.1."""
import math
import os

import numpy as np
import pytest

from oracle import kvq_oracle as O

pytestmark = pytest.mark.cpu


def _h2o_fixture(golden_dir):
    vals = {}
    with open(os.path.join(golden_dir, "h2o_small.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":")
            vals[k.strip()] = [float(x) for x in v.split()]
    return vals


def test_golden_h2o_update(golden_dir):
    f = _h2o_fixture(golden_dir)
    probs = np.array([f["probs0"], f["probs1"]], np.float32)
    kept, cum, ev = O.h2o_accumulate32(probs, np.array(f["retained"], np.int64),
                                       np.array(f["cum"], np.float32), int(f["seq_len"][0]),
                                       int(f["budget"][0]), int(f["n_sink"][0]),
                                       int(f["window"][0]), int(f["new_pos"][0]))
    assert kept.tolist() == [int(x) for x in f["expect_retained"]]
    assert cum.tolist() == f["expect_cum"]
    assert ev.tolist() == [int(x) for x in f["expect_evicted"]]


def _brute_h2o(qs, K, V, T0, steps, budget, ns, w):
    """Independent dict-based H2O: cumulative scores keyed by position."""
    d = K.shape[1]
    keep = list(range(T0))
    cum = {t: 0.0 for t in keep}
    outs = []
    for s in range(steps + 1):
        T = T0 + s
        step_out = []
        for qh in qs[s]:
            sc = {t: sum(float(qh[c]) * float(K[t, c]) for c in range(d)) / math.sqrt(d) for t in keep}
            m = max(sc.values())
            e = {t: math.exp(v - m) for t, v in sc.items()}
            z = sum(e.values())
            for t in keep:
                cum[t] += e[t] / z
            step_out.append([sum(e[t] / z * float(V[t, c]) for t in keep) for c in range(d)])
        outs.append(step_out)
        nxt = T + 1
        while len(keep) > budget - 1:
            cands = [t for t in keep if not (t < ns or t >= nxt - w)]
            if not cands:
                break
            victim = min(cands, key=lambda t: (cum[t], t))
            keep.remove(victim)
            del cum[victim]
        keep.append(T)
        cum[T] = 0.0
    return outs, sorted(keep), cum


def test_h2o_brute_force_three_steps():
    rng = np.random.default_rng(8)
    T0, steps, d, G = 32, 3, 8, 2
    K = rng.standard_normal((T0 + steps + 1, d)).astype(np.float16)
    V = rng.standard_normal((T0 + steps + 1, d)).astype(np.float16)
    qs = (rng.standard_normal((steps + 1, G, d)) * 2).astype(np.float16)
    budget, ns, w = 12, 2, 4
    outs, keep_b, cum_b = _brute_h2o(qs, K, V, T0, steps, budget, ns, w)
    ret = np.arange(T0)
    cum = np.zeros(T0)
    for s in range(steps + 1):
        o, ret, cum, _ = O.h2o_step(qs[s], K, V, ret, cum, T0 + s, budget, ns, w)
        assert np.allclose(o, np.array(outs[s]), atol=1e-12)
    assert sorted(ret.tolist()) == keep_b
    for t, c in zip(ret.tolist(), cum.tolist()):
        assert abs(cum_b[t] - c) < 1e-12


def test_h2o_no_eviction_is_dense_and_mass_is_conserved():
    rng = np.random.default_rng(2)
    T, d, G = 50, 16, 4
    K = rng.standard_normal((T + 1, d)).astype(np.float16)
    V = rng.standard_normal((T + 1, d)).astype(np.float16)
    q = rng.standard_normal((G, d)).astype(np.float16)
    o, ret, cum, ev = O.h2o_step(q, K, V, np.arange(T), np.zeros(T), T, budget=1000,
                                 n_sink=4, window=8)
    assert ev.size == 0 and ret.tolist() == list(range(T + 1))
    for g in range(G):
        ref, _ = O.softmax_attention(q[g].astype(np.float64), K[:T].astype(np.float64),
                                     V[:T].astype(np.float64))
        assert np.array_equal(o[g], ref)
    assert abs(cum.sum() - G) < 1e-12                 # each head's probabilities sum to 1


def test_h2o_protects_sinks_and_window():
    rng = np.random.default_rng(4)
    T, d = 64, 8
    K = rng.standard_normal((T + 1, d)).astype(np.float16)
    V = rng.standard_normal((T + 1, d)).astype(np.float16)
    q = np.zeros((1, d), np.float16)                  # uniform attention
    _, ret, _, ev = O.h2o_step(q, K, V, np.arange(T), np.zeros(T), T, budget=20,
                               n_sink=4, window=8)
    assert set(range(4)) <= set(ret.tolist())
    assert set(range(T + 1 - 8, T + 1)) <= set(ret.tolist())
    # uniform scores: the oldest candidates go first
    assert sorted(ev.tolist()) == list(range(4, 4 + 45))
    assert len(ret) == 20


def test_h2o_fp32_and_fp64_agree_without_ties():
    rng = np.random.default_rng(6)
    T, d, G = 200, 32, 4
    K = rng.standard_normal((T + 1, d)).astype(np.float16)
    V = rng.standard_normal((T + 1, d)).astype(np.float16)
    q = (rng.standard_normal((G, d)) * 3).astype(np.float16)
    ret = np.arange(T)
    _, r64, c64, e64 = O.h2o_step(q, K, V, ret, np.zeros(T), T, 60, 4, 16)
    probs = np.stack([O.sparse_attn(q[g], K, V, ret)[1] for g in range(G)]).astype(np.float32)
    r32, c32, e32 = O.h2o_accumulate32(probs, ret, np.zeros(T, np.float32), T, 60, 4, 16, T)
    assert sorted(r64.tolist()) == sorted(r32.tolist())
    assert np.allclose(c64, c32, atol=1e-6)


# ---------------------------------------------------------------- dense preference

def test_dense_pref_bounds_and_uniform_closed_form():
    rng = np.random.default_rng(0)
    T, d, n_q, k = 300, 128, 8, 16
    K = rng.standard_normal((T, d)).astype(np.float16)
    Q = rng.standard_normal((n_q, d)).astype(np.float16)
    P = O.dense_pref_score(Q, K, k)
    assert 0 <= P <= n_q
    # q = 0: every row is uniform over its L_i = T - n_q + i + 1 keys
    P0 = O.dense_pref_score(np.zeros((n_q, d), np.float16), K, k)
    closed = n_q - sum(min(k, T - n_q + i + 1) / (T - n_q + i + 1) for i in range(n_q))
    assert abs(P0 - closed) < 1e-12


def test_dense_pref_one_hot_and_full_topk():
    rng = np.random.default_rng(1)
    T, d, n_q = 200, 128, 4
    K = rng.standard_normal((T, d)).astype(np.float16)
    # each query aligned, with a large norm, to one key it can see
    Q = np.stack([K[10] * 8 for _ in range(n_q)]).astype(np.float16)
    assert O.dense_pref_score(Q, K, 1) < 1e-6
    assert abs(O.dense_pref_score(Q, K, T)) < 1e-12      # k >= row length: all mass


def test_dense_pref_brute_force():
    rng = np.random.default_rng(2)
    T, d, n_q, k = 20, 8, 5, 3
    K = rng.standard_normal((T, d)).astype(np.float16)
    Q = rng.standard_normal((n_q, d)).astype(np.float16)
    tot = 0.0
    for i in range(n_q):
        L = T - n_q + i + 1
        s = [sum(float(Q[i, c]) * float(K[t, c]) for c in range(d)) / math.sqrt(d) for t in range(L)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = sum(e)
        tot += sum(sorted((x / z for x in e), reverse=True)[:k])
    assert abs(O.dense_pref_score(Q, K, k) - (n_q - tot)) < 1e-12


def test_classify_layer_threshold():
    assert O.classify_layer([10.0, 8.0], 32, 0.2) is True      # mean 9 / 32 = 0.28
    assert O.classify_layer([5.0, 6.0], 32, 0.2) is False      # 0.17
    assert O.classify_layer([6.4, 6.4], 32, 0.2) is False      # equal: not above


def test_classify_heads_per_kv_group():
    """[TailorKV §6] per kv head: the group's mean P / n_q against tau (hand-worked):
    groups (10, 8) -> 0.28 > 0.2 quantize; (5, 6) -> 0.17 sparse; (6.4, 6.4) -> 0.2, not above."""
    P = [10.0, 8.0, 5.0, 6.0, 6.4, 6.4]
    assert O.classify_heads(P, 32, 0.2, 3) == [True, False, False]


def test_classify_heads_reduces_to_the_layer_rule():
    rng = np.random.default_rng(9)
    for _ in range(50):
        P = rng.random(8) * 32
        assert O.classify_heads(P, 32, 0.2, 1) == [O.classify_layer(P, 32, 0.2)]
        # one q head per kv head: each head on its own
        assert O.classify_heads(P, 32, 0.2, 8) == [p / 32 > 0.2 for p in P]
