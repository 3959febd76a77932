"""GPU parity of the sparse-layer path against the oracle:
a4 kv_critical_score (channel lists and fp32 scores bit-exact),
a5 kv_topk_select (index sets bit-exact, including heavy ties),
a6 kv_sparse_attn (outputs <= 2e-3 normwise, probabilities <= 1e-5)."""
import math

import numpy as np
import pytest
import torch

from compressed_kv_cache_quant_gb300 import kvq, synth
from oracle import kvq_oracle as O
from gpu_helpers import ATTN_TOL, attn_err, paged_batch, require_gpu, ws

pytestmark = pytest.mark.gpu


def _fp16_layer(Hq, Hkv, lengths, seed, t_cap=None, extra_pages=3):
    B = len(lengths)
    KV = [synth.kv_rows(T, Hkv, synth.mix(seed, b)) for b, T in enumerate(lengths)]
    n_pages = sum(math.ceil(T / 16) for T in lengths) + extra_pages
    alloc = kvq.Allocator(n_pages, seed=seed % 997 + 1)
    batch, bt = paged_batch(lengths, alloc)
    t_cap = t_cap or (max(lengths) + 7) // 8 * 8
    cache = kvq.LayerCache(Hq, Hkv, 16, n_pages, B, t_cap=t_cap)
    for b, T in enumerate(lengths):
        kvq.kv_quant_pack(cache, batch, b, 0, T, KV[b][0].cuda(), KV[b][1].cuda())
    return cache, batch, bt, KV


def _scores_buf(B, H, max_len):
    stride = (max_len + 7) // 8 * 8
    return torch.full((B, H, stride), float("nan"), device="cuda")


@pytest.mark.parametrize("n_crit", [8, 1, 128])
def test_critical_score_bitexact(n_crit):
    require_gpu()
    Hq, Hkv, lengths = 8, 2, [4096 + 5, 100, 2048]
    cache, batch, bt, KV = _fp16_layer(Hq, Hkv, lengths, synth.mix(synth.BASE_SEED, 10, n_crit))
    B = len(lengths)
    q = synth.queries((B, Hq, 128), synth.mix(synth.BASE_SEED, 11))
    crit = torch.full((B, Hq, n_crit), -1, dtype=torch.int32, device="cuda")
    sc = _scores_buf(B, Hq, batch.max_len)
    kvq.kv_critical_score(cache, batch, q.cuda(), n_crit, crit, sc)
    crit_np, sc_np = crit.cpu().numpy(), sc.cpu().numpy()
    for b, T in enumerate(lengths):
        K = KV[b][0].numpy()
        for h in range(Hq):
            g = O.kv_head_of(h, Hq, Hkv)
            C = O.critical_channels(q[b, h].numpy(), O.key_absmax(K[:, g]), n_crit)
            assert crit_np[b, h].tolist() == C.tolist()
            ref = O.critical_scores(q[b, h].numpy(), K[:, g], C)
            assert np.array_equal(sc_np[b, h, :T].view(np.uint32), ref.view(np.uint32)), (b, h)


def _select(scores_np, lengths, n_heads, k_fixed, ratio, ns, w):
    B = len(lengths)
    max_len = max(lengths)
    stride = scores_np.shape[-1]
    sc = torch.from_numpy(scores_np).cuda()
    seqs = kvq.Batch(torch.zeros((B, math.ceil(max_len / 16)), dtype=torch.int32, device="cuda"),
                     torch.tensor(lengths, dtype=torch.int32, device="cuda"), max_len)
    cap = max(O.topk_count(T, k_fixed if k_fixed >= 0 else O.ratio_k(T, ratio), ns, w) for T in lengths)
    sel = torch.full((B, n_heads, cap), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, n_heads), -7, dtype=torch.int32, device="cuda")
    wk = ws(kvq.kv_topk_select_ws())
    kvq.kv_topk_select(seqs, n_heads, sc, k_fixed, ratio, ns, w, sel, cnt, wk, score_stride=stride)
    kvq.kvq_check(wk)
    return sel.cpu().numpy(), cnt.cpu().numpy()


@pytest.mark.parametrize("lengths,k,ratio,ns,w", [
    ([4096, 300, 37], 128, 0.0, 4, 64),
    ([4096], 0, 0.0, 4, 64),          # sinks + window only: the StreamingLLM mask
    ([100, 196, 197], 128, 0.0, 4, 64),  # T <= n_s + W + k keeps everything
    ([131072 + 17], -1, 0.03, 4, 128),   # ratio mode at 128K
    ([20000, 5], 1000, 0.0, 0, 0),
    ([60000, 131089], -1, 0.03, 4, 128),
    ([5000, 30000], 300, 0.0, 2, 5),      # a window narrower than the cluster
    ([30000], 700, 0.0, 4, 130),          # a window that is not a multiple of 8
    ([20000], 500, 0.0, 4, 600),          # a wide window spanning chunk boundaries
])
def test_topk_select_bitexact_with_ties(lengths, k, ratio, ns, w):
    require_gpu()
    n_heads = 4
    stride = (max(lengths) + 7) // 8 * 8
    rng = np.random.default_rng(sum(lengths) + k)
    scores = np.full((len(lengths), n_heads, stride), np.nan, dtype=np.float32)
    for b, T in enumerate(lengths):
        for h in range(n_heads):
            if h == 0:    # heavy ties: few distinct values
                scores[b, h, :T] = np.round(rng.standard_normal(T) * 2).astype(np.float32)
            elif h == 1:  # all equal, including +0/-0
                scores[b, h, :T] = np.where(rng.random(T) < 0.5, 0.0, -0.0).astype(np.float32)
            elif h == 3:  # moderate ties: a tie group at the k-th value spread over the cluster
                scores[b, h, :T] = (np.round(rng.standard_normal(T) * 64) / 64).astype(np.float32)
            else:
                scores[b, h, :T] = rng.standard_normal(T).astype(np.float32)
    sel, cnt = _select(scores, lengths, n_heads, k, ratio, ns, w)
    for b, T in enumerate(lengths):
        kk = k if k >= 0 else O.ratio_k(T, ratio)
        for h in range(n_heads):
            ref = O.topk_select(scores[b, h, :T], kk, ns, w)
            assert cnt[b, h] == len(ref), (b, h)
            assert sel[b, h, :cnt[b, h]].tolist() == ref.tolist(), (b, h)


def test_sparse_attn_per_q_head_and_probs():
    require_gpu()
    Hq, Hkv, lengths = 8, 2, [4096, 1500]
    cache, batch, bt, KV = _fp16_layer(Hq, Hkv, lengths, synth.mix(synth.BASE_SEED, 20))
    B = len(lengths)
    q = synth.queries((B, Hq, 128), synth.mix(synth.BASE_SEED, 21))
    rng = np.random.default_rng(5)
    cap = 700
    sel = np.zeros((B, Hq, cap), np.int32)
    cnt = np.zeros((B, Hq), np.int32)
    for b, T in enumerate(lengths):
        for h in range(Hq):
            n = int(rng.integers(0, cap + 1)) if h else 0   # head 0: empty list
            ids = np.sort(rng.choice(T, size=min(n, T), replace=False))
            sel[b, h, :len(ids)] = ids
            cnt[b, h] = len(ids)
    out = torch.full((B, Hq, 128), float("nan"), device="cuda")
    probs = torch.full((B, Hq, cap), float("nan"), device="cuda")
    w = ws(kvq.kv_sparse_attn_ws(cache, batch, cap))
    kvq.kv_sparse_attn(cache, batch, q.cuda(), torch.from_numpy(sel).cuda(), torch.from_numpy(cnt).cuda(), 0, out,
                       probs, w)
    kvq.kvq_check(w)
    o, p = out.cpu().numpy(), probs.cpu().numpy()
    for b in range(B):
        for h in range(Hq):
            g = O.kv_head_of(h, Hq, Hkv)
            n = cnt[b, h]
            if n == 0:
                assert np.all(o[b, h] == 0)
                continue
            ref, pr = O.sparse_attn(q[b, h].numpy(), KV[b][0][:, g].numpy(), KV[b][1][:, g].numpy(), sel[b, h, :n])
            assert attn_err(o[b, h], ref) <= ATTN_TOL
            assert np.max(np.abs(p[b, h, :n] - pr)) <= 1e-5


def test_sparse_attn_shared_list_gqa():
    require_gpu()
    Hq, Hkv, T = 8, 2, 3000
    cache, batch, bt, KV = _fp16_layer(Hq, Hkv, [T], synth.mix(synth.BASE_SEED, 22))
    q = synth.queries((1, Hq, 128), synth.mix(synth.BASE_SEED, 23))
    cap = 1200
    rng = np.random.default_rng(8)
    sel = np.zeros((1, Hkv, cap), np.int32)
    cnt = np.array([[cap, 513]], np.int32)
    for g in range(Hkv):
        ids = rng.choice(T, size=cnt[0, g], replace=False)   # unordered list
        sel[0, g, :len(ids)] = ids
    out = torch.empty((1, Hq, 128), device="cuda")
    probs = torch.empty((1, Hq, cap), device="cuda")
    w = ws(kvq.kv_sparse_attn_ws(cache, batch, cap))
    kvq.kv_sparse_attn(cache, batch, q.cuda(), torch.from_numpy(sel).cuda(), torch.from_numpy(cnt).cuda(), 1, out,
                       probs, w)
    kvq.kvq_check(w)
    o, p = out.cpu().numpy(), probs.cpu().numpy()
    for h in range(Hq):
        g = O.kv_head_of(h, Hq, Hkv)
        n = cnt[0, g]
        ref, pr = O.sparse_attn(q[0, h].numpy(), KV[0][0][:, g].numpy(), KV[0][1][:, g].numpy(), sel[0, g, :n])
        assert attn_err(o[0, h], ref) <= ATTN_TOL
        assert np.max(np.abs(p[0, h, :n] - pr)) <= 1e-5


def test_sparse_layer_pipeline_config_tiny():
    """Tiny single layer as a sparse layer: 8 critical channels, top-128 +
    4 sinks + 64 window, exact attention on the selection (T=4096, GQA 4)."""
    require_gpu()
    Hq, Hkv, T = 8, 2, 4096
    cache, batch, bt, KV = _fp16_layer(Hq, Hkv, [T], synth.mix(synth.BASE_SEED + 0, 30))
    q = synth.queries((1, Hq, 128), synth.mix(synth.BASE_SEED + 0, 31))
    sc = _scores_buf(1, Hq, T)
    crit = torch.empty((1, Hq, 8), dtype=torch.int32, device="cuda")
    kvq.kv_critical_score(cache, batch, q.cuda(), 8, crit, sc)
    cap = 128 + 4 + 64
    sel = torch.empty((1, Hq, cap), dtype=torch.int32, device="cuda")
    cnt = torch.empty((1, Hq), dtype=torch.int32, device="cuda")
    wk = ws(kvq.kv_topk_select_ws())
    kvq.kv_topk_select(batch, Hq, sc, 128, 0.0, 4, 64, sel, cnt, wk)
    out = torch.empty((1, Hq, 128), device="cuda")
    w = ws(kvq.kv_sparse_attn_ws(cache, batch, cap))
    kvq.kv_sparse_attn(cache, batch, q.cuda(), sel, cnt, 0, out, None, w)
    kvq.kvq_check(w)
    kvq.kvq_check(wk)
    K, V = KV[0][0].numpy(), KV[0][1].numpy()
    for h in range(Hq):
        g = O.kv_head_of(h, Hq, Hkv)
        C = O.critical_channels(q[0, h].numpy(), O.key_absmax(K[:, g]), 8)
        a = O.critical_scores(q[0, h].numpy(), K[:, g], C)
        ids = O.topk_select(a, 128, 4, 64)
        assert cnt[0, h].item() == len(ids) == cap
        assert sel[0, h].cpu().numpy().tolist() == ids.tolist()
        ref, _ = O.sparse_attn(q[0, h].numpy(), K[:, g], V[:, g], ids)
        assert attn_err(out[0, h].cpu().numpy(), ref) <= ATTN_TOL


def test_sparse_attn_flags_bad_index():
    require_gpu()
    cache, batch, bt, KV = _fp16_layer(4, 2, [100], 5)
    sel = torch.tensor([[[3, 500]] * 4], dtype=torch.int32, device="cuda")
    cnt = torch.tensor([[2] * 4], dtype=torch.int32, device="cuda")
    out = torch.empty((1, 4, 128), device="cuda")
    w = ws(kvq.kv_sparse_attn_ws(cache, batch, 2))
    kvq.kv_sparse_attn(cache, batch, torch.zeros((1, 4, 128), dtype=torch.float16, device="cuda"), sel, cnt, 0,
                       out, None, w)
    with pytest.raises(kvq.KvqError):
        kvq.kvq_check(w)
    # the valid row alone determines the output
    assert torch.allclose(out[0, 0].cpu().float(), KV[0][1][3, 0].float(), atol=1e-6)


@pytest.mark.parametrize("use_hist,lengths,k,ratio,ns,w", [
    (True, [4096 + 3, 1000], -1, 0.03, 4, 128),
    (True, [4096], 128, 0.0, 4, 64),
    (False, [3000, 300], 128, 0.0, 4, 64),
    (True, [150], 128, 0.0, 4, 64),     # everything kept
])
def test_fused_append_score_select_attn(use_hist, lengths, k, ratio, ns, w):
    """kv_append_critical_score + kv_select_sparse_attn (the fused two-launch
    sparse-layer step) against the oracle: the newest token is appended, the
    scores, the selection and the attention over it match."""
    require_gpu()
    Hq, Hkv = 8, 2
    B = len(lengths)
    seed = synth.mix(synth.BASE_SEED, 60, int(use_hist), k)
    full = [T + 2 for T in lengths]
    cache, batch, bt, KV = _fp16_layer(Hq, Hkv, full, seed)
    # the cache holds T - 1 tokens before the step; rebuild it with the first T - 1 only
    cache2 = kvq.LayerCache(Hq, Hkv, 16, cache.num_blocks, B, t_cap=cache.t_cap)
    lens_before = [T - 1 for T in lengths]
    batch2 = kvq.Batch(batch.block_table, torch.tensor(lens_before, dtype=torch.int32, device="cuda"), batch.max_len)
    for b, T in enumerate(lengths):
        kvq.kv_quant_pack(cache2, batch2, b, 0, T - 1, KV[b][0][:T - 1].cuda(), KV[b][1][:T - 1].cuda())
    kvq.kvq_seq_lens_add(batch2.seq_lens, 1)
    kn = torch.stack([KV[b][0][T - 1] for b, T in enumerate(lengths)]).cuda()
    vn = torch.stack([KV[b][1][T - 1] for b, T in enumerate(lengths)]).cuda()
    q = synth.queries((B, Hq, 128), synth.mix(seed, 1))
    sc = _scores_buf(B, Hq, batch2.max_len)
    hist = torch.zeros((B, Hq, 4096), dtype=torch.int32, device="cuda") if use_hist else None
    wa = ws(kvq.kv_append_critical_score_ws())
    kvq.kv_append_critical_score(cache2, batch2, kn, vn, q.cuda(), 8, None, sc, hist, ns, w, wa)
    cap = max(O.topk_count(T, k if k >= 0 else O.ratio_k(T, ratio), ns, w) for T in lengths)
    sel = torch.full((B, Hq, cap), -1, dtype=torch.int32, device="cuda")
    cnt = torch.zeros((B, Hq), dtype=torch.int32, device="cuda")
    out = torch.full((B, Hq, 128), float("nan"), device="cuda")
    wsx = ws(kvq.kv_select_sparse_attn_ws())
    kvq.kv_select_sparse_attn(cache2, batch2, q.cuda(), sc, hist, k, ratio, ns, w, sel, cnt, out, wsx)
    kvq.kvq_check(wa)
    kvq.kvq_check(wsx)
    if use_hist:
        assert int(hist.abs().sum().item()) == 0     # cleared for the next layer
    sc_np, sel_np, cnt_np, o = sc.cpu().numpy(), sel.cpu().numpy(), cnt.cpu().numpy(), out.cpu().numpy()
    am = cache2.k_absmax.cpu().numpy()
    for b, T in enumerate(lengths):
        K, V = KV[b][0][:T].numpy(), KV[b][1][:T].numpy()
        kk = k if k >= 0 else O.ratio_k(T, ratio)
        for h in range(Hq):
            g = O.kv_head_of(h, Hq, Hkv)
            assert np.array_equal(am[b, g], O.key_absmax(K[:, g]).astype(np.float32))
            C = O.critical_channels(q[b, h].numpy(), O.key_absmax(K[:, g]), 8)
            a = O.critical_scores(q[b, h].numpy(), K[:, g], C)
            assert np.array_equal(sc_np[b, h, :T].view(np.uint32), a.view(np.uint32)), (b, h)
            ids = O.topk_select(a, kk, ns, w)
            assert cnt_np[b, h] == len(ids)
            assert sel_np[b, h, :len(ids)].tolist() == ids.tolist(), (b, h)
            ref, _ = O.sparse_attn(q[b, h].numpy(), K[:, g], V[:, g], ids)
            assert attn_err(o[b, h], ref) <= ATTN_TOL, (b, h)
    # the appended rows are in the pages and the channel-major copy
    for b, T in enumerate(lengths):
        p = T - 1
        for g in range(Hkv):
            assert np.array_equal(cache2.k16[bt[b, p // 16], g, p % 16].cpu().numpy(), KV[b][0][p, g].numpy())
            assert np.array_equal(cache2.v16[bt[b, p // 16], g, p % 16].cpu().numpy(), KV[b][1][p, g].numpy())
            assert np.array_equal(cache2.kT[b, g, :, p].cpu().numpy(), KV[b][0][p, g].numpy())
