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


# ---- f1 block-granular selection   [Meeting §8.1, block pruning]

@pytest.mark.parametrize("T,k", [(50, 10), (97, 33), (300, 40)])
def test_block_select_of_single_tokens_is_topk(T, k):
    """With one-token blocks the block mean is the token's own score, so block
    pruning must pick exactly what the independent token top-K picks."""
    s = np.random.default_rng(T).standard_normal(T).astype(np.float32)
    assert T > 4 + 16 + k
    got = O.block_select(s, k, 4, 16, 1)
    assert got.tolist() == O.topk_select(s, k, 4, 16).tolist()


def test_block_importance_closed_form():
    """Scores t (exact in fp32): a block's importance is the midpoint of its
    candidate range; blocks inside the sinks or the window are -inf."""
    T, B, ns, W = 200, 16, 20, 40
    imp = O.block_importance(np.arange(T, dtype=np.float32), ns, W, B)
    assert len(imp) == 13
    for j in range(13):
        lo, hi = max(j * B, ns), min((j + 1) * B, T - W)
        if lo < hi:
            assert imp[j] == np.float32((lo + hi - 1) / 2)
        else:
            assert imp[j] == -np.inf
    # block 0 lies in the sinks; T - W = 160 ends the candidates with block 9 = [144, 160)
    assert imp[0] == -np.inf and imp[1] == np.float32(25.5) and imp[9] == np.float32(151.5)
    assert np.all(imp[10:] == -np.inf)


def test_block_select_constant_scores_keep_the_first_blocks():
    T, B, ns, W, n = 1000, 64, 4, 128, 3
    got = O.block_select(np.full(T, 0.25, np.float32), n, ns, W, B)
    want = sorted(set(range(0, 3 * B)) | set(range(T - W, T)))
    assert got.tolist() == want


def test_block_select_planted_block_and_ties():
    T, B = 640, 64
    s = np.zeros(T, np.float32)
    s[5 * B:6 * B] = 1.0          # the planted block wins
    s[2 * B:3 * B:2] = 0.5        # blocks 2 and 7 tie at a mean of 0.25 ...
    s[7 * B + 1:8 * B:2] = 0.5    # ... with different contents: the lower block goes first
    got = O.block_select(s, 2, 0, 0, B)
    assert got.tolist() == list(range(2 * B, 3 * B)) + list(range(5 * B, 6 * B))


@pytest.mark.parametrize("seed", range(6))
def test_block_select_brute_force_invariant(seed):
    """Small integer scores (exact means as fractions): the kept blocks are the
    n best by (mean desc, block asc); every kept block beats every other block
    that has candidates, and sinks/window are always kept."""
    from fractions import Fraction
    rng = np.random.default_rng(100 + seed)
    T, B, ns, W = int(rng.integers(20, 60)), 8, int(rng.integers(0, 6)), int(rng.integers(0, 9))
    s = rng.integers(-3, 4, size=T).astype(np.float32)
    nb = -(-T // B)
    n = int(rng.integers(0, nb + 1))
    got = set(O.block_select(s, n, ns, W, B).tolist())
    keyed = []
    for j in range(nb):
        lo, hi = max(j * B, ns), min((j + 1) * B, T - W)
        m = Fraction(int(sum(int(x) for x in s[lo:hi])), hi - lo) if lo < hi else None
        keyed.append((m, j))
    ranked = sorted(keyed, key=lambda mj: (mj[0] is None, -(mj[0] or 0), mj[1]))
    want = set(range(min(ns, T))) | set(range(max(T - W, 0), T))
    for _, j in ranked[:n]:
        want |= set(range(j * B, min((j + 1) * B, T)))
    assert got == want


def test_block_count():
    assert O.block_count(131072, 0.03, 64) == 61
    assert O.block_count(4096, 0.03, 64) == 1
    assert O.block_count(100, 0.5, 64) == 1


@pytest.mark.parametrize("case", ["normal", "critical_scores", "ties", "near_ties"])
def test_block_mean_fp32_agrees_with_exact_mean_except_near_ties(case):
    """The block importance is an fp32 mean (the scores' own precision, summed in a
    fixed order).  Against the exact mean (a rational number, here in fp64 over
    fp32 inputs, whose error is far below 1e-5 relative), the kept blocks are the
    same except where the two blocks exchanged at the cut have exact means within
    1e-5 relative of each other -- the near-tie allowance of the selection."""
    rng = np.random.default_rng({"normal": 1, "critical_scores": 2, "ties": 3, "near_ties": 4}[case])
    for rep in range(20):
        T, B = int(rng.integers(2000, 9000)), int(rng.choice([16, 64, 128]))
        ns, W = 4, 128
        if case == "normal":
            s = rng.standard_normal(T).astype(np.float32)
        elif case == "critical_scores":  # sums of 8 products of fp16 values, like the critical scores
            q = rng.standard_normal(8).astype(np.float16).astype(np.float32)
            K = (rng.standard_normal((T, 8)) * np.where(rng.random(8) < 0.5, 10, 1)).astype(np.float16)
            s = np.zeros(T, np.float32)
            for c in range(8):
                s = s + q[c] * K[:, c].astype(np.float32)
        elif case == "ties":  # whole blocks repeat: many exactly equal means
            base = rng.standard_normal(B).astype(np.float32)
            s = np.tile(base, -(-T // B))[:T] * rng.choice([1.0, 1.0, 0.5], size=-(-T // B)).repeat(B)[:T]
            s = s.astype(np.float32)
        else:  # a block whose mean differs from another's by a rounding or two
            s = rng.standard_normal(T).astype(np.float32)
            j0, j1 = 3, 7
            s[j1 * B:(j1 + 1) * B] = s[j0 * B:(j0 + 1) * B][::-1]
        nb = -(-T // B)
        n = int(rng.integers(1, max(2, nb // 3)))
        imp32 = O.block_importance(s, ns, W, B)
        exact = np.full(nb, -np.inf)
        for j in range(nb):
            lo, hi = max(j * B, ns), min((j + 1) * B, T - W)
            if lo < hi:
                exact[j] = float(np.sum(s[lo:hi].astype(np.float64))) / (hi - lo)
        keep32 = set(np.lexsort((np.arange(nb), -imp32.astype(np.float64)))[:n].tolist())
        keep64 = set(np.lexsort((np.arange(nb), -exact))[:n].tolist())
        assert set(O.block_select(s, n, ns, W, B).tolist()) >= {t for j in keep32 for t in range(j * B, min((j + 1) * B, T))}
        only32, only64 = keep32 - keep64, keep64 - keep32
        assert len(only32) == len(only64)
        for a in only32:
            for b in only64:
                assert abs(exact[a] - exact[b]) <= 1e-5 * max(abs(exact[a]), abs(exact[b])), (case, rep, a, b)


# ---- f1 selection shared by the query heads of a kv head (GQA)   [TailorKV §2.3 per kv head]

def _golden_group(golden_dir):
    rows = {}
    with open(os.path.join(golden_dir, "group_select_small.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = [c.strip() for c in line.split("|")]
                rows[k] = [float(x) for x in v.split()]
    return rows


def test_golden_group_selection(golden_dir):
    g = _golden_group(golden_dir)
    q = np.array([g["q0"], g["q1"]], dtype=np.float16)
    K = np.array([g["K0"], g["K1"], g["K2"], g["K3"]], dtype=np.float16).T      # [T][d]
    C = O.group_critical_channels(q, O.key_absmax(K), int(g["n_crit"][0]))
    assert C.tolist() == [int(x) for x in g["channels"]]
    s = O.group_critical_scores(q, K, C)
    assert s.tolist() == g["scores"]
    ns, w, k = [int(x) for x in g["n_sink window k"]]
    assert O.topk_select(s, k, ns, w).tolist() == [int(x) for x in g["selected"]]


@pytest.mark.parametrize("seed", range(4))
def test_group_of_one_is_the_per_head_definition(seed):
    """A group of one query head reduces to the per-head channels and scores, bit for bit."""
    rng = np.random.default_rng(30 + seed)
    K = (rng.standard_normal((500, 128)) * np.where(rng.random(128) < 0.05, 10, 1)).astype(np.float16)
    q = rng.standard_normal(128).astype(np.float16)
    am = O.key_absmax(K)
    C = O.critical_channels(q, am, 8)
    assert O.group_critical_channels(q[None], am, 8).tolist() == C.tolist()
    assert np.array_equal(O.group_critical_scores(q[None], K, C).view(np.uint32),
                          O.critical_scores(q, K, C).view(np.uint32))


def test_group_scores_on_all_channels_are_the_summed_dot_products():
    """With every channel critical, the group score is sum_h q_h . K_t, up to fp32 rounding."""
    rng = np.random.default_rng(41)
    K = rng.standard_normal((300, 128)).astype(np.float16)
    q = rng.standard_normal((4, 128)).astype(np.float16)
    C = O.group_critical_channels(q, O.key_absmax(K), 128)
    assert C.tolist() == list(range(128))
    s = O.group_critical_scores(q, K, C).astype(np.float64)
    exact = (K.astype(np.float64) @ q.astype(np.float64).T).sum(axis=1)
    bound = (np.abs(K.astype(np.float64)) @ np.abs(q.astype(np.float64)).T).sum(axis=1) * 128 * 2.0 ** -24
    assert np.all(np.abs(s - exact) <= bound)


@pytest.mark.parametrize("seed", range(6))
def test_group_channels_brute_force(seed):
    """Small integer queries (exact sums): the chosen channels are the n_crit best by
    (sum_h |q_h,c| * max|K_c| desc, channel asc), computed with Python integers."""
    rng = np.random.default_rng(50 + seed)
    G, d, n = int(rng.integers(1, 5)), 16, int(rng.integers(1, 9))
    q = rng.integers(-3, 4, size=(G, d)).astype(np.float16)
    am = rng.integers(0, 5, size=d).astype(np.float16)
    got = O.group_critical_channels(q, am, n).tolist()
    imp = [(sum(abs(int(q[h, c])) for h in range(G)) * int(am[c]), c) for c in range(d)]
    want = sorted(c for _, c in sorted(imp, key=lambda ic: (-ic[0], ic[1]))[:n])
    assert got == want
