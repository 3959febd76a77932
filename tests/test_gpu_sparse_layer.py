"""GPU parity of kv_sparse_layer_decode (append + critical scores + top-K
selection + attention of a sparse layer in one launch) against the oracle:
appended rows and fp32 scores bit-exact, selection bit-exact, attention
within 2e-3 normwise.
Sources: TailorKV §2.3, §5.1; KV-cache survey §一.1, §三.1; meeting article §3.2."""
import math

import numpy as np
import pytest
import torch

from compressed_kv_cache_quant_gb300 import kvq, synth
from oracle import kvq_oracle as O
from gpu_helpers import ATTN_TOL, attn_err, paged_batch, require_gpu, ws

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("Hq,Hkv,lengths,n_crit,k,ratio,ns,w", [
    (8, 2, [4096], 8, 128, 0.0, 4, 64),              # the tiny single-layer configuration
    (8, 2, [4096 + 3, 1000, 150], 8, -1, 0.03, 4, 128),
    (4, 4, [20000], 16, 500, 0.0, 2, 32),
    (32, 8, [131072 + 5], 8, -1, 0.03, 4, 128),      # 128K context, ratio 0.03
])
def test_sparse_layer_decode_matches_oracle(Hq, Hkv, lengths, n_crit, k, ratio, ns, w):
    require_gpu()
    B = len(lengths)
    seed = synth.mix(synth.BASE_SEED + 1, 70, Hq, n_crit, sum(lengths))
    KV = [synth.kv_rows(T, Hkv, synth.mix(seed, b)) for b, T in enumerate(lengths)]
    n_pages = sum(math.ceil(T / 16) for T in lengths) + 4
    alloc = kvq.Allocator(n_pages, seed=seed % 1009 + 1)
    batch, bt = paged_batch(lengths, alloc, lengths=[T - 1 for T in lengths])
    t_cap = (max(lengths) + 7) // 8 * 8
    cache = kvq.LayerCache(Hq, Hkv, 16, n_pages, B, t_cap=t_cap)
    for b, T in enumerate(lengths):
        kvq.kv_quant_pack(cache, batch, b, 0, T - 1, KV[b][0][:T - 1].cuda(), KV[b][1][:T - 1].cuda())
    kvq.kvq_seq_lens_add(batch.seq_lens, 1)
    kn = torch.stack([KV[b][0][T - 1] for b, T in enumerate(lengths)]).cuda()
    vn = torch.stack([KV[b][1][T - 1] for b, T in enumerate(lengths)]).cuda()
    q = synth.queries((B, Hq, 128), synth.mix(seed, 1))
    stride = (batch.max_len + 7) // 8 * 8
    sc = torch.full((B, Hq, stride), float("nan"), device="cuda")
    cap = max(O.topk_count(T, k if k >= 0 else O.ratio_k(T, ratio), ns, w) for T in lengths)
    sel = torch.full((B, Hq, cap), -1, dtype=torch.int32, device="cuda")
    cnt = torch.zeros((B, Hq), dtype=torch.int32, device="cuda")
    out = torch.full((B, Hq, 128), float("nan"), device="cuda")
    wk = ws(kvq.kv_sparse_layer_decode_ws())
    kvq.kv_sparse_layer_decode(cache, batch, kn, vn, q.cuda(), n_crit, k, ratio, ns, w, out, wk, scores=sc, sel=sel,
                               sel_count=cnt)
    kvq.kvq_check(wk)
    sc_np, sel_np, cnt_np, o = sc.cpu().numpy(), sel.cpu().numpy(), cnt.cpu().numpy(), out.cpu().numpy()
    for b, T in enumerate(lengths):
        K, V = KV[b][0][:T].numpy(), KV[b][1][:T].numpy()
        kk = k if k >= 0 else O.ratio_k(T, ratio)
        heads = range(Hq) if Hq <= 8 else [0, 1, 5, 13, 31]
        for h in heads:
            g = O.kv_head_of(h, Hq, Hkv)
            C = O.critical_channels(q[b, h].numpy(), O.key_absmax(K[:, g]), n_crit)
            a = O.critical_scores(q[b, h].numpy(), K[:, g], C)
            assert np.array_equal(sc_np[b, h, :T].view(np.uint32), a.view(np.uint32)), (b, h)
            ids = O.topk_select(a, kk, ns, w)
            assert cnt_np[b, h] == len(ids)
            assert sel_np[b, h, :len(ids)].tolist() == ids.tolist(), (b, h)
            ref, _ = O.sparse_attn(q[b, h].numpy(), K[:, g], V[:, g], ids)
            assert attn_err(o[b, h], ref) <= ATTN_TOL, (b, h)
        p = T - 1
        for g in range(Hkv):
            assert np.array_equal(cache.k16[bt[b, p // 16], g, p % 16].cpu().numpy(), KV[b][0][p, g].numpy())
            assert np.array_equal(cache.v16[bt[b, p // 16], g, p % 16].cpu().numpy(), KV[b][1][p, g].numpy())
            assert np.array_equal(cache.kT[b, g, :, p].cpu().numpy(), KV[b][0][p, g].numpy())
            assert np.array_equal(cache.k_absmax[b, g].cpu().numpy(), O.key_absmax(K[:, g]).astype(np.float32))


def test_sparse_layer_decode_without_optional_outputs_is_the_same():
    """The bench path (no score copy, no selection output) gives the same attention."""
    require_gpu()
    Hq, Hkv, T = 8, 2, 5000
    seed = synth.mix(synth.BASE_SEED + 1, 71)
    K, V = synth.kv_rows(T, Hkv, seed)
    alloc = kvq.Allocator(math.ceil(T / 16) + 1, seed=2)
    outs = []
    for opt in (True, False):
        batch, bt = paged_batch([T], kvq.Allocator(math.ceil(T / 16) + 1, seed=2), lengths=[T - 1])
        cache = kvq.LayerCache(Hq, Hkv, 16, math.ceil(T / 16) + 1, 1, t_cap=(T + 7) // 8 * 8)
        kvq.kv_quant_pack(cache, batch, 0, 0, T - 1, K[:T - 1].cuda(), V[:T - 1].cuda())
        kvq.kvq_seq_lens_add(batch.seq_lens, 1)
        q = synth.queries((1, Hq, 128), synth.mix(seed, 1)).cuda()
        out = torch.empty((1, Hq, 128), device="cuda")
        wk = ws(kvq.kv_sparse_layer_decode_ws())
        extra = {}
        if opt:
            extra = dict(scores=torch.empty((1, Hq, (T + 7) // 8 * 8), device="cuda"),
                         sel=torch.empty((1, Hq, 300), dtype=torch.int32, device="cuda"),
                         sel_count=torch.empty((1, Hq), dtype=torch.int32, device="cuda"))
        kvq.kv_sparse_layer_decode(cache, batch, K[T - 1][None].cuda(), V[T - 1][None].cuda(), q, 8, 128, 0.0, 4,
                                   64, out, wk, **extra)
        kvq.kvq_check(wk)
        outs.append(out.cpu().numpy())
    del alloc
    for h in range(Hq):
        assert attn_err(outs[1][0, h], outs[0][0, h]) <= 1e-5


@pytest.mark.parametrize("n_crit,T,k,expect_radix", [
    (8, 40000, 600, False),   # many tie at the k-th key: third digit pass, the cut inside one CTA
    (2, 40000, 6000, True),   # thousands tie: distributed radix passes after the early attention
])
def test_sparse_layer_bench_path_ties(n_crit, T, k, expect_radix):
    """Integer keys in {-1, 0, 1} and a unit query: the approximate scores tie in bulk, the
    kept set follows the lower-position rule at the k-th key, and the one-pass path's early
    attention over the rows kept for certain plus the attention over the rest equals the
    oracle (TailorKV §2.3; KV-cache survey §三.1)."""
    require_gpu()
    Hq, Hkv, ns, w = 8, 2, 4, 64
    seed = synth.mix(synth.BASE_SEED + 1, 302, n_crit, k)
    g = torch.Generator().manual_seed(seed)
    K = torch.randint(-1, 2, (T, Hkv, 128), generator=g).to(torch.float16)
    V = synth.normal((T, Hkv, 128), synth.mix(seed, 2))
    n_pages = math.ceil(T / 16) + 2
    alloc = kvq.Allocator(n_pages, seed=7)
    batch, bt = paged_batch([T], alloc, lengths=[T - 1])
    cache = kvq.LayerCache(Hq, Hkv, 16, n_pages, 1, t_cap=(T + 7) // 8 * 8)
    kvq.kv_quant_pack(cache, batch, 0, 0, T - 1, K[:T - 1].cuda(), V[:T - 1].cuda())
    kvq.kvq_seq_lens_add(batch.seq_lens, 1)
    q = torch.ones((1, Hq, 128), dtype=torch.float16)
    out = torch.full((1, Hq, 128), float("nan"), device="cuda")
    wk = ws(kvq.kv_sparse_layer_decode_ws())
    kvq.kv_sparse_layer_decode(cache, batch, K[T - 1][None].cuda(), V[T - 1][None].cuda(), q.cuda(), n_crit, k, 0.0,
                               ns, w, out, wk)
    kvq.kvq_check(wk)
    listed, compacted, radix, _ = kvq.kvq_read_path_counters(wk)
    assert (radix > 0) == expect_radix
    o = out.cpu().numpy()
    Kn, Vn = K.numpy(), V.numpy()
    for h in range(Hq):
        gk = O.kv_head_of(h, Hq, Hkv)
        C = O.critical_channels(q[0, h].numpy(), O.key_absmax(Kn[:, gk]), n_crit)
        ids = O.topk_select(O.critical_scores(q[0, h].numpy(), Kn[:, gk], C), k, ns, w)
        ref, _ = O.sparse_attn(q[0, h].numpy(), Kn[:, gk], Vn[:, gk], ids)
        assert attn_err(o[0, h], ref) <= ATTN_TOL, h
