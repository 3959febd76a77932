"""GPU parity of f1 kv_block_select (block pruning of the meeting article, §8.1)
against the oracle: kept token sets and counts bit-exact (block importances are
fp32 sums in ascending order and an fp32 division on both sides), ties to the lower
block, ragged lengths, tiny and 128K contexts; and the whole block-sparse
pipeline (critical scores -> block selection -> exact attention) against the
oracle's."""
import math

import numpy as np
import pytest
import torch

from compressed_kv_cache_quant_gb300 import kvq, synth
from oracle import kvq_oracle as O
from gpu_helpers import ATTN_TOL, attn_err, paged_batch, require_gpu, ws

pytestmark = pytest.mark.gpu


def _block_select(scores_np, lengths, n_heads, n_keep, ratio, ns, w, block, cap=None):
    B = len(lengths)
    max_len = max(lengths)
    stride = scores_np.shape[-1]
    sc = torch.from_numpy(scores_np).cuda()
    seqs = kvq.Batch(torch.zeros((B, math.ceil(max_len / 16)), dtype=torch.int32, device="cuda"),
                     torch.tensor(lengths, dtype=torch.int32, device="cuda"), max_len)
    cap = cap or max(lengths)
    sel = torch.full((B, n_heads, cap), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, n_heads), -7, dtype=torch.int32, device="cuda")
    wk = ws(kvq.kv_block_select_ws(seqs, n_heads, block))
    kvq.kv_block_select(seqs, n_heads, sc, n_keep, ratio, ns, w, block, sel, cnt, wk, score_stride=stride)
    kvq.kvq_check(wk)
    return sel.cpu().numpy(), cnt.cpu().numpy()


@pytest.mark.parametrize("lengths,n_keep,ratio,ns,w,block", [
    ([4096, 300, 37], 3, 0.0, 4, 64, 64),
    ([131072 + 17], -1, 0.03, 4, 128, 64),   # the 128K layer: 61 blocks of 64
    ([60000, 131089], -1, 0.03, 4, 128, 128),
    ([5000, 1000, 70], -1, 0.1, 0, 0, 16),   # page-sized blocks, no sinks or window
    ([100, 20, 3], 2, 0.0, 4, 64, 64),       # contexts inside the sinks and window
    ([20000], 0, 0.0, 4, 64, 64),            # no block kept: the StreamingLLM mask
    ([9000, 4097], 1000, 0.0, 70, 33, 64),   # more blocks asked than exist; odd sink and window
])
def test_block_select_bitexact_with_ties(lengths, n_keep, ratio, ns, w, block):
    require_gpu()
    n_heads = 3
    stride = (max(lengths) + 7) // 8 * 8
    rng = np.random.default_rng(sum(lengths) + block)
    scores = np.full((len(lengths), n_heads, stride), np.nan, dtype=np.float32)
    for b, T in enumerate(lengths):
        scores[b, 0, :T] = np.round(rng.standard_normal(T) * 2).astype(np.float32)  # many equal block means
        scores[b, 1, :T] = rng.standard_normal(T).astype(np.float32)
        scores[b, 2, :T] = np.where(rng.random(T) < 0.5, 1.0, -0.0).astype(np.float32)
        scores[b, 2, :T:block * 3] = 0.0  # equal-mean blocks next to different ones
    sel, cnt = _block_select(scores, lengths, n_heads, n_keep, ratio, ns, w, block)
    for b, T in enumerate(lengths):
        n = n_keep if n_keep >= 0 else O.block_count(T, ratio, block)
        for h in range(n_heads):
            ref = O.block_select(scores[b, h, :T], n, ns, w, block)
            assert cnt[b, h] == len(ref), (b, h)
            assert sel[b, h, :cnt[b, h]].tolist() == ref.tolist(), (b, h)


def test_block_select_cut_at_capacity_flags_overflow():
    require_gpu()
    T = 4096
    scores = np.random.default_rng(3).standard_normal((1, 1, T)).astype(np.float32)
    with pytest.raises(kvq.KvqError):
        _block_select(scores, [T], 1, 10, 0.0, 4, 64, 64, cap=300)


def test_block_sparse_pipeline_matches_oracle():
    """Critical scores -> block selection -> exact attention, per q head."""
    require_gpu()
    Hq, Hkv, lengths, block, ratio = 8, 2, [8192 + 9, 3000], 64, 0.05
    B = len(lengths)
    seed = synth.mix(synth.BASE_SEED, 1500)
    KV = [synth.kv_rows(T, Hkv, synth.mix(seed, b)) for b, T in enumerate(lengths)]
    n_pages = sum(math.ceil(T / 16) for T in lengths) + 3
    batch, bt = paged_batch(lengths, kvq.Allocator(n_pages, seed=7))
    cache = kvq.LayerCache(Hq, Hkv, 16, n_pages, B, t_cap=(max(lengths) + 7) // 8 * 8)
    for b, T in enumerate(lengths):
        kvq.kv_quant_pack(cache, batch, b, 0, T, KV[b][0].cuda(), KV[b][1].cuda())
    q = synth.queries((B, Hq, 128), synth.mix(seed, 99))
    crit = torch.zeros((B, Hq, 8), dtype=torch.int32, device="cuda")
    stride = (batch.max_len + 7) // 8 * 8
    sc = torch.full((B, Hq, stride), float("nan"), device="cuda")
    kvq.kv_critical_score(cache, batch, q.cuda(), 8, crit, sc)
    cap = batch.max_len
    sel = torch.zeros((B, Hq, cap), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((B, Hq), dtype=torch.int32, device="cuda")
    wk = ws(kvq.kv_block_select_ws(batch, Hq, block))
    kvq.kv_block_select(batch, Hq, sc, -1, ratio, 4, 64, block, sel, cnt, wk)
    out = torch.full((B, Hq, 128), float("nan"), device="cuda")
    wa = ws(kvq.kv_sparse_attn_ws(cache, batch, cap))
    kvq.kv_sparse_attn(cache, batch, q.cuda(), sel, cnt, 0, out, None, wa)
    kvq.kvq_check(wk)
    kvq.kvq_check(wa)
    o, s_np, c_np = out.cpu().numpy(), sel.cpu().numpy(), cnt.cpu().numpy()
    for b, T in enumerate(lengths):
        K, V = KV[b][0].numpy(), KV[b][1].numpy()
        for h in range(Hq):
            g = O.kv_head_of(h, Hq, Hkv)
            C = O.critical_channels(q[b, h].numpy(), O.key_absmax(K[:, g]), 8)
            a = O.critical_scores(q[b, h].numpy(), K[:, g], C)
            ids = O.block_select(a, O.block_count(T, ratio, block), 4, 64, block)
            assert s_np[b, h, :c_np[b, h]].tolist() == ids.tolist(), (b, h)
            ref, _ = O.sparse_attn(q[b, h].numpy(), K[:, g], V[:, g], ids)
            assert attn_err(o[b, h], ref) <= ATTN_TOL, (b, h)
