"""Plain CPU oracle for compressed-KV decode attention.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check of
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import or run
anything in this directory.  The GPU library never imports it and it imports
nothing from the GPU library; the two share no code.  Inputs reach both sides
from the seeded generators, which hold none of the method's arithmetic.

Every function works on logical (unpaged) arrays: one sequence, one kv head,
tokens in order.  Paging, packing bit order and GPU memory layout are
implementation details of the GPU library and do not appear here.

Sources (the pages this method is read from; a citation names the page and
the section on it):

* [TailorKV] "TailorKV" article, ijyty.com/news/1204784 -- §2.1 dense
  preference score, §2.2 1-bit quantization of quantization-friendly layers
  (the ``quant_1bit`` snippet), §2.3 dynamic loading of sparsity-friendly
  layers (critical channels, approximate scores, top-K), §5.1 configuration
  (sparse_ratio, critical_channels).
* [KVSurvey] "大语言模型长上下文推理与KV Cache前沿压缩策略解析",
  bbs.huaweicloud.com/blogs/490932 -- §一 PagedAttention (16-token blocks,
  shared blocks), §三.1 StreamingLLM sinks + window, §三.2 H2O cumulative
  attention scores.
* [OnDevice] "端侧大模型KV缓存量化卸载协同：详解分层稀疏注意力与异构内存池动态迁移机制",
  ufo.work/2026/495 -- §3.1 K per-channel asymmetric INT4/INT8, V grouped
  (group 32/64), §3.2 fused dequant -> QK^T -> softmax -> PV.
* [Meeting] "长上下文会议大模型推理KV缓存稀疏化与量化联合压缩：剖析重要性评分指标与异构内存分层调度策略",
  ufo.work/2026/545 -- §3.2 softmax attention over retained tokens, §4.2
  double-buffered prefetch, §8.1 block-sparse decode attention.

Precision: the quantizer runs in IEEE fp32 (inputs are fp16 widened to fp32;
round half to even), because its output is an integer code that both sides
must decide in the same precision.  Attention, softmax and the dense
preference score run in fp64.  The critical-channel score runs in fp32 in a
fixed summation order (ascending channel), because it decides an integer
(the top-K index set).

Readings of points the pages leave open are marked READING below; the full
list lives in the design notes of the repository.

Parity pins: every function here is pinned by tests under ``tests/`` that
check it against closed forms, invariants, brute force on tiny inputs and
hand-worked fixtures in ``tests/golden/``.  No function is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

HEAD_DIM = 128
K_GROUP_TOKENS = 64


# ---------------------------------------------------------------------------
# a1: asymmetric min/max b-bit quantization   [TailorKV §2.2; OnDevice §3.1]
# ---------------------------------------------------------------------------

def quantize_groups(x16, bits):
    """Quantize every group (the LAST axis of ``x16``) to ``bits``-bit codes.

    [TailorKV §2.2] per group: scale = (max - min) / (2^b - 1), zero = min,
    code = clamp(round((x - zero) / scale), 0, 2^b - 1); scale and zero are
    stored as fp16.

    READING: ``round`` is round-half-to-even (the snippet calls torch.round);
    the code is computed with the unrounded fp32 scale and only the stored
    scale is rounded to fp16 (the snippet divides first and converts the
    scale to fp16 on return); a group with max == min gets scale 0 and all
    codes 0 (the snippet would divide by zero).

    Returns (codes int64, scale16 float16, zero16 float16, scale32 float32);
    scale/zero have the group axis removed.
    """
    x = np.asarray(x16, dtype=np.float16).astype(np.float32)
    levels = np.float32(2 ** bits - 1)
    mn = x.min(axis=-1, keepdims=True)
    mx = x.max(axis=-1, keepdims=True)
    scale32 = (mx - mn) / levels                      # fp32, one rounding
    ok = scale32 > 0
    safe = np.where(ok, scale32, np.float32(1.0))
    with np.errstate(over="ignore", invalid="ignore"):
        u = (x - mn) / safe                           # fp32, two roundings
    codes = np.clip(np.rint(u), np.float32(0), levels)
    codes = np.where(ok, codes, np.float32(0)).astype(np.int64)
    with np.errstate(over="ignore"):
        scale16 = scale32[..., 0].astype(np.float16)
    zero16 = mn[..., 0].astype(np.float16)            # exact: min of fp16 values
    return codes, scale16, zero16, scale32[..., 0]


def pack_k(k16, bits, group_tokens=K_GROUP_TOKENS):
    """Quantize the keys of one (sequence, kv head): K is [T][d] fp16.

    [TailorKV §2.2] keys are quantized per channel; [OnDevice §3.1] per
    channel asymmetric with a zero point; the group runs over ``group_tokens``
    consecutive tokens (64, [TailorKV §2.2 snippet and §5.2]).

    READING: tokens past the last complete 64-token group (the "tail") stay
    in fp16 and are attended exactly; they are quantized once the group fills.

    Returns dict(codes [n_full*64][d] int64, scale16/zero16/scale32 [n_groups][d],
    tail [T - n_full*64][d] fp16, n_packed).
    """
    k16 = np.asarray(k16, dtype=np.float16)
    T, d = k16.shape
    n_groups = T // group_tokens
    n_packed = n_groups * group_tokens
    g = k16[:n_packed].reshape(n_groups, group_tokens, d).transpose(0, 2, 1)  # [g][c][t]
    codes, s16, z16, s32 = quantize_groups(g, bits)
    codes = codes.transpose(0, 2, 1).reshape(n_packed, d)
    return dict(codes=codes, scale16=s16, zero16=z16, scale32=s32,
                tail=k16[n_packed:].copy(), n_packed=n_packed, bits=bits,
                group_tokens=group_tokens)


def pack_v(v16, bits, group_dims):
    """Quantize the values of one (sequence, kv head): V is [T][d] fp16.

    [TailorKV §2.2] values are quantized per token; [OnDevice §3.1] in groups
    of ``group_dims`` (32 or 64) consecutive channels of head_dim.

    Returns dict(codes [T][d] int64, scale16/zero16/scale32 [T][d/group_dims]).
    """
    v16 = np.asarray(v16, dtype=np.float16)
    T, d = v16.shape
    assert d % group_dims == 0
    g = v16.reshape(T, d // group_dims, group_dims)
    codes, s16, z16, s32 = quantize_groups(g, bits)
    return dict(codes=codes.reshape(T, d), scale16=s16, zero16=z16, scale32=s32,
                bits=bits, group_dims=group_dims)


def quantize_groups_sym(x16, bits):
    """Symmetric quantization of every group (the LAST axis of ``x16``).

    [On-device article §3.1: V quantized INT4 symmetric, in groups of 32/64
    channels] per group: scale = max |x| / L, code = clamp(round(x / scale), -L, L)
    with L = 2^(b-1) - 1; the scale is stored as fp16.

    READING: the restricted symmetric range -L..L (no -2^(b-1)), round half to
    even, IEEE fp32 arithmetic on the fp16 inputs and codes computed with the
    fp32 scale as in ``quantize_groups``; an all-zero group gets scale 0 and codes
    0; b >= 2 (for b = 1 the range is empty).
    Returns (codes int64 in [-L, L], scale16 float16, scale32 float32)."""
    assert bits >= 2
    x = np.asarray(x16, dtype=np.float16).astype(np.float32)
    L = np.float32(2 ** (bits - 1) - 1)
    amax = np.abs(x).max(axis=-1, keepdims=True)
    scale32 = (amax / L).astype(np.float32)           # fp32, one rounding
    ok = scale32 > 0
    safe = np.where(ok, scale32, np.float32(1.0))
    with np.errstate(over="ignore", invalid="ignore"):
        u = (x / safe).astype(np.float32)             # fp32, one rounding
    codes = np.clip(np.rint(u), -L, L)
    codes = np.where(ok, codes, np.float32(0)).astype(np.int64)
    return codes, scale32[..., 0].astype(np.float16), scale32[..., 0]


def pack_v_sym(v16, bits, group_dims):
    """Symmetric quantization of the values of one (sequence, kv head), per token
    in groups of ``group_dims`` channels [on-device article §3.1].
    Returns dict(codes [T][d] int64 in [-L, L], scale16/scale32 [T][d/group_dims])."""
    v16 = np.asarray(v16, dtype=np.float16)
    T, d = v16.shape
    g = v16.reshape(T, d // group_dims, group_dims)
    codes, s16, s32 = quantize_groups_sym(g, bits)
    return dict(codes=codes.reshape(T, d), scale16=s16, scale32=s32, bits=bits, group_dims=group_dims,
                symmetric=True)


def channel_variance(k16):
    """[Meeting §8.2] per-channel variance of fp16 keys [T][d], order-independent:
    every fp16 value is an integer multiple of 2^-24, so the sums S1 = sum_t K_t,c
    (in units of 2^-24) and S2 = sum_t K_t,c^2 (in units of 2^-48) are formed
    exactly as integers, each rounded once to fp64 (round to nearest even), and
    Var_c = (S2 - S1^2 / T) / T follows in fp64 with one rounding per operation.
    S2 is summed in three int64 parts of the 40-bit magnitude u = a 2^20 + b
    (u^2 = a^2 2^40 + 2ab 2^20 + b^2), exact for T <= 2^22."""
    K = np.asarray(k16, dtype=np.float16)
    T = K.shape[0]
    assert T <= 1 << 22
    x = (K.astype(np.float64) * 2.0 ** 24).astype(np.int64)       # exact: |x| < 2^40
    s1 = x.sum(axis=0)
    u = np.abs(x)
    a, b = u >> 20, u & ((1 << 20) - 1)
    p2, p1, p0 = (a * a).sum(axis=0), (2 * a * b).sum(axis=0), (b * b).sum(axis=0)
    var = np.empty(K.shape[1], dtype=np.float64)
    for c in range(K.shape[1]):
        S1 = float(int(s1[c])) * 2.0 ** -24                          # Python int -> float rounds to nearest even
        S2 = float((int(p2[c]) << 40) + (int(p1[c]) << 20) + int(p0[c])) * 2.0 ** -48
        var[c] = (S2 - S1 * S1 / T) / T if T else 0.0
    return var


def outlier_channels(k16, n_out):
    """[Meeting §8.2] outlier channels of one (sequence, kv head): the channels of
    largest variance.  READING (the page calibrates offline on 1000 samples; here
    the prompt itself is the calibration set, as the on-device article's online
    calibration from prefill statistics, §3.2): Var_c from ``channel_variance``;
    the n_out largest, ties -> lower channel, returned ascending.  The page's
    "top 0.5 %" of a 128-channel head is n_out = ceil(0.005 * 128) = 1."""
    var = channel_variance(k16)
    order = np.lexsort((np.arange(var.shape[0]), -var))
    return np.sort(order[:n_out])


def pack_k_outlier(k16, bits, out_ch, group_tokens=K_GROUP_TOKENS):
    """[Meeting §8.2] keys with outlier channels isolated: the main cache is
    ``pack_k`` with the outlier channels' codes, scale and zero set to 0 (they
    contribute nothing there); the outlier channels of the packed tokens are kept
    as fp16 in a side cache (``outlier_values`` [n_packed][n_out]).  READING: the
    page's main cache is "INT4 ... symmetric ... scale, zero_point" (a
    contradiction); the main cache here is the K quantizer of this library
    (asymmetric, per channel), unchanged for the normal channels."""
    pk = pack_k(k16, bits, group_tokens)
    out_ch = np.asarray(out_ch, dtype=np.int64)
    n = pk["n_packed"]
    pk["codes"][:, out_ch] = 0
    pk["scale16"][:, out_ch] = 0
    pk["zero16"][:, out_ch] = 0
    pk["scale32"][:, out_ch] = 0
    pk["outliers"] = out_ch
    pk["outlier_values"] = np.asarray(k16, dtype=np.float16)[:n][:, out_ch].copy()
    return pk


def dequant_k(pk):
    """fp64 keys as the quantized cache represents them: zero + code * scale
    for packed tokens (stored fp16 scale/zero), fp16 values for the tail and,
    with isolated outlier channels (``pack_k_outlier``), for those channels."""
    n_packed = pk["n_packed"]
    gt = pk["group_tokens"]
    d = pk["tail"].shape[1]
    out = np.empty((n_packed + pk["tail"].shape[0], d), dtype=np.float64)
    if n_packed:
        grp = np.arange(n_packed) // gt
        out[:n_packed] = (pk["zero16"].astype(np.float64)[grp]
                          + pk["codes"].astype(np.float64) * pk["scale16"].astype(np.float64)[grp])
        if "outliers" in pk:
            out[:n_packed, pk["outliers"]] = pk["outlier_values"].astype(np.float64)
    out[n_packed:] = pk["tail"].astype(np.float64)
    return out


def dequant_v(pv):
    """fp64 values as the quantized cache represents them: zero + code * scale,
    or code * scale for a symmetric cache (``pack_v_sym``)."""
    T, d = pv["codes"].shape
    gd = pv["group_dims"]
    j = np.arange(d) // gd
    vals = pv["codes"].astype(np.float64) * pv["scale16"].astype(np.float64)[:, j]
    if pv.get("symmetric"):
        return vals
    return pv["zero16"].astype(np.float64)[:, j] + vals


# ---------------------------------------------------------------------------
# f4: FP8 E4M3 KV cache   [meeting article §6 item 2: FP8 E4M3 preferred over INT4
# where the hardware has it -- no dequantization arithmetic]
# ---------------------------------------------------------------------------

def fp8_e4m3_decode(codes):
    """Values of E4M3 bytes: sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
    exponent 0 holds the subnormals m * 2^-9; S.1111.111 is NaN; no infinities.
    Returns float64 (exact)."""
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    sgn = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sgn * val


def fp8_e4m3_encode(x16):
    """fp16 -> E4M3 byte, round to nearest with ties to even mantissa, finite
    values beyond the largest (448) saturate to +-448.  READING: the pages name
    the format (E4M3) but no scale; K and V are cast directly, one byte per value
    (fp16 inputs here stay within the range).  Integer arithmetic on the fp16
    value: for |x| in the normal range of E4M3 the significand keeps 3 fraction
    bits, below 2^-6 the grid is 2^-9.  Returns uint8 codes."""
    x = np.asarray(x16, dtype=np.float16).astype(np.float64)
    sign = (np.signbit(x)).astype(np.int64) << 7
    nan = np.isnan(x)
    a = np.where(nan, 0.0, np.minimum(np.abs(x), 512.0))   # inf saturates like any |x| > 448
    with np.errstate(divide="ignore", invalid="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0))).astype(np.int64)
    e = np.clip(e, -6, 8)                      # the binade's exponent; below 2^-6 the subnormal grid 2^-9
    ulp = np.exp2((e - 3).astype(np.float64))  # 3 fraction bits
    q = a / ulp                                # exact: a is fp16, ulp a power of two
    lo = np.floor(q)
    frac = q - lo
    up = (frac > 0.5) | ((frac == 0.5) & (lo.astype(np.int64) % 2 == 1))
    n = (lo + up).astype(np.int64)             # multiple of ulp after rounding
    mag = n * ulp                              # the rounded magnitude
    # re-encode the magnitude (a carry may have moved it to the next binade)
    sub = mag < 2.0 ** -6
    code_sub = np.round(mag / 2.0 ** -9).astype(np.int64)
    with np.errstate(divide="ignore", invalid="ignore"):
        e2 = np.floor(np.log2(np.where(mag > 0, mag, 1.0))).astype(np.int64)
    m2 = np.round((mag / np.exp2(e2.astype(np.float64)) - 1.0) * 8).astype(np.int64)
    code_norm = ((e2 + 7) << 3) | m2
    out = np.where(sub, code_sub, code_norm)
    out = np.where(mag > 448.0, 0x7E, out)     # saturate (finite)
    out = np.where(nan, 0x7F, out)
    return (out | sign).astype(np.uint8)


def fp8_attention(q16, k16, v16):
    """Exact softmax attention (fp64) of one query over a cache stored as E4M3:
    keys and values are the decoded E4M3 values of the fp16 rows."""
    K = fp8_e4m3_decode(fp8_e4m3_encode(k16))
    V = fp8_e4m3_decode(fp8_e4m3_encode(v16))
    return softmax_attention(np.asarray(q16, dtype=np.float16), K, V)


# ---------------------------------------------------------------------------
# exact softmax attention (shared definition used by a3, a6, a7, a8)
# [Meeting §3.2: Softmax(Q K_ret^T / sqrt(d)) V_ret; OnDevice §3.2]
# ---------------------------------------------------------------------------

def softmax_attention(q, K, V):
    """One query against n keys: s = K q / sqrt(d), p = softmax(s), o = p V.
    fp64 throughout; the max is subtracted before exponentiation.
    Returns (o [d], p [n])."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    s = (K @ q) / math.sqrt(q.shape[0])
    e = np.exp(s - s.max())
    p = e / e.sum()
    return p @ V, p


def kv_head_of(h, n_q_heads, n_kv_heads):
    """GQA: q head h reads kv head floor(h * H_kv / H_q)."""
    return (h * n_kv_heads) // n_q_heads


# ---------------------------------------------------------------------------
# a3: decode attention over the quantized cache   [OnDevice §3.2; TailorKV §2.2]
# ---------------------------------------------------------------------------

def decode_attn_quant(q16, packed_k, packed_v):
    """Decode attention of every q head of one sequence over its quantized
    cache.  ``q16`` is [H_q][d]; ``packed_k``/``packed_v`` are lists (one per
    kv head) of ``pack_k``/``pack_v`` results.  Packed keys are dequantized,
    tail keys are used as fp16, values are always dequantized.
    Returns o [H_q][d] fp64."""
    q16 = np.asarray(q16, dtype=np.float16)
    Hq, d = q16.shape
    Hkv = len(packed_k)
    out = np.empty((Hq, d), dtype=np.float64)
    cache = {}
    for h in range(Hq):
        g = kv_head_of(h, Hq, Hkv)
        if g not in cache:
            cache[g] = (dequant_k(packed_k[g]), dequant_v(packed_v[g]))
        Kh, Vh = cache[g]
        out[h], _ = softmax_attention(q16[h].astype(np.float64), Kh, Vh)
    return out


# ---------------------------------------------------------------------------
# a4: critical channels and approximate scores   [TailorKV §2.3]
# ---------------------------------------------------------------------------

def critical_channels(q16, absmax16, n_crit):
    """[TailorKV §2.3] channel importance s_i = |q_i| * max_t |K_{t,i}|; the
    n_crit most important channels (ties -> lower channel) are returned in
    ascending channel order.  fp64 (exact for fp16 inputs)."""
    q = np.abs(np.asarray(q16, dtype=np.float16).astype(np.float64))
    a = np.asarray(absmax16, dtype=np.float64)
    s = q * a
    idx = np.arange(s.shape[0])
    order = np.lexsort((idx, -s))        # primary: s descending, then index
    return np.sort(order[:n_crit])


def key_absmax(k16):
    """max_t |K_{t,c}| over all cached tokens, per channel (fp16, exact)."""
    return np.abs(np.asarray(k16, dtype=np.float16)).max(axis=0)


def critical_scores(q16, k16, channels):
    """[TailorKV §2.3] approximate attention score of every cached token from
    the critical channels only: a_t = sum_{c in C} q_c K_{t,c}.
    READING: fp32, summed over C in ascending channel order starting from +0.
    Returns float32 [T]."""
    q = np.asarray(q16, dtype=np.float16).astype(np.float32)
    K = np.asarray(k16, dtype=np.float16)
    acc = np.zeros(K.shape[0], dtype=np.float32)
    for c in np.sort(np.asarray(channels)):
        acc = acc + q[c] * K[:, c].astype(np.float32)
    return acc


# ---------------------------------------------------------------------------
# f1: selection shared by the query heads of one kv head (GQA)
# [TailorKV §2.3 applied per kv head; meeting article §8.1 item 1]
# ---------------------------------------------------------------------------

def group_critical_channels(q16_group, absmax16, n_crit):
    """Critical channels shared by the G query heads ``q16_group`` [G][d] of one
    kv head.  READING (the pages say only "the query"): a channel's importance
    for the kv head is the sum over the group's heads of |q_h,c| -- an fp32 sum
    in ascending head order -- times max_t |K_t,c| (fp32); the n_crit most
    important channels, ties -> lower channel, in ascending order.  fp32 in a
    fixed order because it decides an integer (the channel set).  With G = 1
    this is ``critical_channels``."""
    q = np.abs(np.asarray(q16_group, dtype=np.float16).astype(np.float32))
    s = q[0].copy()
    for h in range(1, q.shape[0]):
        s = (s + q[h]).astype(np.float32)
    s = (s * np.asarray(absmax16, dtype=np.float16).astype(np.float32)).astype(np.float32)
    idx = np.arange(s.shape[0])
    order = np.lexsort((idx, -s.astype(np.float64)))
    return np.sort(order[:n_crit])


def group_critical_scores(q16_group, k16, channels):
    """Approximate score of every cached token for the G query heads of one kv
    head.  READING: each head's approximate score on the shared channels
    (``critical_scores``: fp32, ascending channel) summed over the heads in
    ascending order in fp32.  Returns float32 [T]."""
    q16_group = np.asarray(q16_group, dtype=np.float16)
    tot = critical_scores(q16_group[0], k16, channels)
    for h in range(1, q16_group.shape[0]):
        tot = (tot + critical_scores(q16_group[h], k16, channels)).astype(np.float32)
    return tot


# ---------------------------------------------------------------------------
# a5: top-K selection with sinks and a recent window
# [TailorKV §2.3 top-K, §5.1 sparse_ratio; KVSurvey §三.1 sinks + window]
# ---------------------------------------------------------------------------

def topk_select(scores, k, n_sink, window):
    """Selected token ids (ascending) for one query head.

    Tokens [0, n_sink) (attention sinks) and [T - window, T) (recent window)
    are always kept; among the rest the k highest scores are added, ties ->
    lower index.  If the sinks, window and k cover everything, all tokens are
    selected."""
    scores = np.asarray(scores, dtype=np.float32)
    T = scores.shape[0]
    if T <= n_sink + window + k:
        return np.arange(T, dtype=np.int64)
    cand = np.arange(n_sink, T - window)
    order = np.lexsort((cand, -scores[cand].astype(np.float64)))
    top = cand[order[:k]]
    keep = np.concatenate([np.arange(n_sink), top, np.arange(T - window, T)])
    return np.sort(keep).astype(np.int64)


def topk_count(T, k, n_sink, window):
    """Number of ids ``topk_select`` returns for a length-T sequence."""
    return T if T <= n_sink + window + k else n_sink + window + k


def ratio_k(T, ratio):
    """K from a retention ratio: floor(ratio * T) ([TailorKV §5.1] sparse_ratio)."""
    return int(math.floor(ratio * T))


# ---------------------------------------------------------------------------
# a6: exact attention over a selected token set   [Meeting §3.2, §8.1]
# ---------------------------------------------------------------------------

def sparse_attn(q16, k16, v16, ids):
    """Exact softmax attention of one fp16 query over the fp16 K/V rows
    ``ids``.  Returns (o [d] fp64, p [len(ids)] fp64) with p in ``ids`` order."""
    ids = np.asarray(ids, dtype=np.int64)
    K = np.asarray(k16, dtype=np.float16)[ids]
    V = np.asarray(v16, dtype=np.float16)[ids]
    return softmax_attention(np.asarray(q16, dtype=np.float16), K, V)


# ---------------------------------------------------------------------------
# a7: H2O cumulative attention accumulate / evict   [KVSurvey §三.2, §三.1]
# ---------------------------------------------------------------------------

def h2o_protected(pos, next_len, n_sink, window):
    """A retained token is never evicted while it is a sink or sits in the
    recent window of the next step (positions >= next_len - window)."""
    pos = np.asarray(pos)
    return (pos < n_sink) | (pos >= next_len - window)


def h2o_evict(retained, cum, next_len, budget_after, n_sink, window):
    """Evict unprotected tokens, lowest (cum, position) first, until at most
    ``budget_after`` remain (or nothing unprotected is left).
    READING: ties on the cumulative score evict the older token first.
    Returns (kept positions, kept cum, evicted positions), keeping input order."""
    retained = np.asarray(retained, dtype=np.int64)
    cum = np.asarray(cum)
    excess = retained.shape[0] - budget_after
    if excess <= 0:
        return retained, cum, np.empty(0, dtype=np.int64)
    prot = h2o_protected(retained, next_len, n_sink, window)
    cand = np.nonzero(~prot)[0]
    order = np.lexsort((retained[cand], cum[cand].astype(np.float64)))
    drop = cand[order[:excess]]
    mask = np.ones(retained.shape[0], dtype=bool)
    mask[drop] = False
    return retained[mask], cum[mask], retained[drop]


def h2o_accumulate32(probs32, retained, cum32, seq_len, budget, n_sink, window,
                     new_pos):
    """One accumulate/evict/admit update on fp32 state, for one (sequence, kv head).

    ``probs32`` [G][n] fp32: this step's attention probability of every
    retained token for each of the G query heads sharing the kv head.
    cum += (((p_0 + p_1) + p_2) + ...) in fp32 (heads in ascending order, the
    sum added to cum last).  Then unprotected tokens are evicted (lowest cum,
    then lowest position) down to budget - 1 when a new token will be
    admitted (``new_pos`` >= 0), else down to budget; the new token joins with
    cum 0.  The window is taken relative to the next step's length
    seq_len + 1.  Returns (retained, cum32, evicted)."""
    probs32 = np.asarray(probs32, dtype=np.float32)
    inc = probs32[0].copy()
    for g in range(1, probs32.shape[0]):
        inc = inc + probs32[g]
    cum = np.asarray(cum32, dtype=np.float32) + inc
    after = budget - 1 if new_pos >= 0 else budget
    kept, kcum, ev = h2o_evict(retained, cum, seq_len + 1, after, n_sink, window)
    if new_pos >= 0:
        kept = np.concatenate([kept, [new_pos]])
        kcum = np.concatenate([kcum, np.zeros(1, dtype=np.float32)])
    return kept, kcum.astype(np.float32), ev


def h2o_step(q16_group, k16, v16, retained, cum, seq_len, budget, n_sink, window,
             admit_next=True):
    """One H2O decode step in fp64 for one (sequence, kv head).

    The G query heads of the group attend the retained tokens (positions
    < seq_len; the newest token was admitted by the previous step); their
    probabilities, summed over the group, are added to the cumulative scores
    (a heavy-hitter score per kv head -- READING for GQA); then the lowest
    unprotected tokens are evicted and position ``seq_len`` (the next token)
    is admitted with score 0.  The first call, with every token retained and
    cum 0, is the initial heavy-hitter selection over the prompt.
    Returns (o [G][d], retained, cum, evicted)."""
    q16_group = np.asarray(q16_group, dtype=np.float16)
    G = q16_group.shape[0]
    retained = np.asarray(retained, dtype=np.int64)
    outs = []
    inc = np.zeros(retained.shape[0], dtype=np.float64)
    for g in range(G):
        o, p = sparse_attn(q16_group[g], k16, v16, retained)
        outs.append(o)
        inc += p
    cum = np.asarray(cum, dtype=np.float64) + inc
    after = budget - 1 if admit_next else budget
    kept, kcum, ev = h2o_evict(retained, cum, seq_len + 1, after, n_sink, window)
    if admit_next:
        kept = np.concatenate([kept, [seq_len]])
        kcum = np.concatenate([kcum, [0.0]])
    return np.stack(outs), kept, kcum, ev


# ---------------------------------------------------------------------------
# a8: dense-preference score and layer classification   [TailorKV §2.1]
# ---------------------------------------------------------------------------

def dense_pref_score(q16_recent, k16, topk):
    """[TailorKV §2.1] P = n_q - sum over the top-k entries of every row of
    A = softmax(Q K^T / sqrt(d_h)) for the n_q most recent queries of one head.

    READING: the queries sit at the last n_q positions and attend causally
    (query i at position T - n_q + i sees keys 0..T - n_q + i); a row shorter
    than k contributes all of its entries.  fp64."""
    Q = np.asarray(q16_recent, dtype=np.float16).astype(np.float64)
    K = np.asarray(k16, dtype=np.float16).astype(np.float64)
    n_q, d = Q.shape
    T = K.shape[0]
    total = 0.0
    for i in range(n_q):
        L = T - n_q + i + 1
        s = (K[:L] @ Q[i]) / math.sqrt(d)
        e = np.exp(s - s.max())
        p = e / e.sum()
        kk = min(topk, L)
        total += np.sort(p)[L - kk:].sum()
    return n_q - total


def classify_layer(P_heads, n_q, tau):
    """[TailorKV §2.1] READING of the comparison lost in the page text: a
    layer is quantization-friendly when its dense-preference score, averaged
    over heads and normalised by n_q, exceeds tau (dense attention -> large
    P -> quantize; sparse attention -> small P -> top-K)."""
    return float(np.mean(P_heads)) / n_q > tau


def classify_heads(P_heads, n_q, tau, n_kv_heads):
    """[TailorKV §6: the layer-level strategy carried down to attention heads]
    READING: the unit that is quantized or made sparse is a kv head's cache, so a
    kv head is quantization-friendly when the dense-preference score averaged over
    the q heads sharing it (ascending head order, fp64) and normalised by n_q
    exceeds tau -- ``classify_layer`` applied to each group of q heads.  With one
    kv head this is the layer rule.  Returns a list of bools, one per kv head."""
    P = np.asarray(P_heads, dtype=np.float64)
    G = P.shape[0] // n_kv_heads
    return [classify_layer(P[g * G:(g + 1) * G], n_q, tau) for g in range(n_kv_heads)]


# ---------------------------------------------------------------------------
# a9: offload gather   [Meeting §4.2 double buffer; TailorKV §2.3, §3.1]
# ---------------------------------------------------------------------------

def offload_gather(rows16, ids):
    """The rows ``ids`` of a host-resident fp16 [T][d] array, in ``ids`` order,
    as raw bytes: what the host-link gather must deliver into HBM."""
    rows16 = np.asarray(rows16, dtype=np.float16)
    out = np.empty((len(ids), rows16.shape[1]), dtype=np.float16)
    for i, t in enumerate(ids):
        out[i] = rows16[int(t)]
    return out


# ---------------------------------------------------------------------------
# f1: block-granular selection   [Meeting §8.1, item 1: block pruning]
# ---------------------------------------------------------------------------

def block_importance(scores, n_sink, window, block):
    """[Meeting §8.1] importance of every ``block``-token block (block j holds
    tokens [j*block, (j+1)*block) clipped to T): the mean of the approximate
    scores of its candidate tokens (n_sink <= t < T - window).  READING: the
    page asks for the block mean but fixes no arithmetic; it is taken in the
    scores' own precision, an fp32 sum in ascending t divided by the
    candidate count in fp32, in that fixed order because the importance
    decides an integer (the kept blocks).  A block without candidates gets
    -inf.  Returns fp32 [ceil(T / block)]."""
    scores = np.asarray(scores, dtype=np.float32)
    T = scores.shape[0]
    nb = -(-T // block)
    imp = np.full(nb, -np.inf, dtype=np.float32)
    for j in range(nb):
        lo, hi = max(j * block, n_sink), min((j + 1) * block, T - window)
        if lo < hi:
            s = np.float32(0.0)
            for t in range(lo, hi):  # plain left-to-right fp32 sum
                s = np.float32(s + scores[t])
            imp[j] = np.float32(s / np.float32(hi - lo))
    return imp


def block_select(scores, n_keep, n_sink, window, block):
    """[Meeting §8.1] Selected token ids (ascending) with block pruning: the
    sinks [0, n_sink) and the window [T - window, T) as in ``topk_select``, plus
    every token of the ``n_keep`` blocks of highest importance (ties -> lower
    block; blocks without candidates rank last, at -inf).  READING: the page
    keeps the "top P%" of blocks; n_keep = floor(P * ceil(T / block)) is
    ``block_count``."""
    scores = np.asarray(scores, dtype=np.float32)
    T = scores.shape[0]
    imp = block_importance(scores, n_sink, window, block)
    order = np.lexsort((np.arange(len(imp)), -imp.astype(np.float64)))
    keep = np.zeros(T, dtype=bool)
    keep[:min(n_sink, T)] = True
    keep[max(T - window, 0):] = True
    for j in order[:n_keep]:
        keep[j * block:min((j + 1) * block, T)] = True
    return np.nonzero(keep)[0].astype(np.int64)


def block_count(T, ratio, block):
    """Blocks kept at retention ratio P: floor(P * ceil(T / block))."""
    return int(math.floor(ratio * float(-(-T // block))))
