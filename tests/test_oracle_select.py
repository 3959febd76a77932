"""Pins for the oracle's critical-channel scoring (a4) and token selection
(a5): hand-worked fixtures, brute-force sorts, the StreamingLLM mask and
the full-channel reduction.
Sources: TailorKV §2.3 and §5.1; KV-cache survey §三.1."""
import os

import numpy as np
import pytest

from oracle import kvq_oracle as O

pytestmark = pytest.mark.cpu


def _topk_cases(golden_dir):
    out = []
    with open(os.path.join(golden_dir, "topk_small.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            ns, w, k, sc, ex = [c.strip() for c in line.split("|")]
            out.append((int(ns), int(w), int(k), [float(v) for v in sc.split()],
                        [int(v) for v in ex.split()]))
    return out


def test_golden_topk(golden_dir):
    cases = _topk_cases(golden_dir)
    assert len(cases) >= 5
    for ns, w, k, sc, ex in cases:
        got = O.topk_select(np.array(sc, np.float32), k, ns, w)
        assert got.tolist() == ex, (ns, w, k)
        assert len(got) == O.topk_count(len(sc), k, ns, w)


@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force(seed):
    rng = np.random.default_rng(seed)
    T = int(rng.integers(1, 60))
    ns, w, k = int(rng.integers(0, 5)), int(rng.integers(0, 9)), int(rng.integers(0, 20))
    sc = np.round(rng.standard_normal(T) * 3).astype(np.float32)     # many ties
    got = O.topk_select(sc, k, ns, w)
    if T <= ns + w + k:
        assert got.tolist() == list(range(T))
        return
    cand = sorted(range(ns, T - w), key=lambda t: (-float(sc[t]), t))[:k]
    want = sorted(set(range(ns)) | set(cand) | set(range(T - w, T)))
    assert got.tolist() == want


def test_topk_zero_is_streaming_mask():
    T, ns, w = 500, 4, 64
    sc = np.random.default_rng(0).standard_normal(T).astype(np.float32)
    got = O.topk_select(sc, 0, ns, w)
    mask = [t for t in range(T) if t < ns or t >= T - w]
    assert got.tolist() == mask


def test_topk_all_equal_takes_lowest():
    got = O.topk_select(np.ones(100, np.float32), 10, 4, 8)
    assert got.tolist() == list(range(14)) + list(range(92, 100))


def test_ratio_k():
    assert O.ratio_k(131072, 0.03) == 3932
    assert O.ratio_k(131136, 0.03) == 3934


def test_critical_channels_brute_force_and_ties():
    rng = np.random.default_rng(3)
    for _ in range(20):
        q = rng.standard_normal(128).astype(np.float16)
        a = np.abs(rng.standard_normal(128) * np.where(rng.random(128) < 0.05, 10, 1)).astype(np.float16)
        got = O.critical_channels(q, a, 8)
        s = [(-(abs(float(q[c])) * float(a[c])), c) for c in range(128)]
        want = sorted(c for _, c in sorted(s)[:8])
        assert got.tolist() == want
    # ties -> lower channel
    assert O.critical_channels(np.ones(128, np.float16), np.ones(128, np.float16), 8).tolist() == list(range(8))
    # a channel with zero query weight never beats a non-zero one
    q = np.zeros(128, np.float16)
    q[[5, 70]] = 1
    assert O.critical_channels(q, np.ones(128, np.float16), 2).tolist() == [5, 70]


def test_key_absmax():
    K = np.array([[1, -3], [-2, 2]], np.float16)
    assert O.key_absmax(K).tolist() == [2, 3]


def test_critical_scores_full_channels_is_dot():
    rng = np.random.default_rng(5)
    q = rng.standard_normal(128).astype(np.float16)
    K = rng.standard_normal((200, 128)).astype(np.float16)
    a = O.critical_scores(q, K, np.arange(128))
    exact = K.astype(np.float64) @ q.astype(np.float64)
    bound = 128 * 2.0 ** -24 * (np.abs(K.astype(np.float64)) @ np.abs(q.astype(np.float64)))
    assert np.all(np.abs(a.astype(np.float64) - exact) <= bound)
    assert a.dtype == np.float32


def test_critical_scores_order_is_ascending_channel():
    """(2^24 + 1) - 2^24 = 0 in fp32 when summed in channel order 0,1,2 from +0;
    any other order gives 1."""
    q = np.zeros(128, np.float16)
    K = np.zeros((1, 128), np.float16)
    q[[0, 1, 2]] = [4096, 1, -4096]
    K[0, [0, 1, 2]] = [4096, 1, 4096]
    assert O.critical_scores(q, K, [2, 0, 1])[0] == 0.0
    # a score built only from -0 products is +0 (sum starts at +0)
    q2 = np.zeros(128, np.float16)
    q2[0] = -1
    K2 = np.zeros((1, 128), np.float16)
    v = O.critical_scores(q2, K2, [0])[0]
    assert v == 0.0 and not np.signbit(v)


def test_offload_gather_bytes():
    rng = np.random.default_rng(0)
    rows = rng.standard_normal((50, 128)).astype(np.float16)
    ids = [49, 0, 7, 7, 13]
    got = O.offload_gather(rows, ids)
    assert got.tobytes() == b"".join(rows[i].tobytes() for i in ids)
