"""GPU parity of the selection shared by the query heads of a kv head (GQA):
kv_group_critical_score (channels and fp32 scores bit-exact), kv_topk_select
over the kv heads' scores (bit-exact), and kv_sparse_attn with one list per kv
head (within 2e-3 normwise) against the oracle.
Sources: TailorKV §2.3, §5.1 (applied per kv head); KV-cache survey §三.1;
meeting article §3.2, §8.1."""
import math

import numpy as np
import pytest
import torch

from compressed_kv_cache_quant_gb300 import kvq, synth
from oracle import kvq_oracle as O
from gpu_helpers import ATTN_TOL, attn_err, paged_batch, require_gpu, ws

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("Hq,Hkv,lengths,n_crit,k,ratio,ns,w", [
    (8, 2, [4096], 8, 128, 0.0, 4, 64),                  # the tiny configuration's shape, GQA 4
    (16, 2, [5000 + 3, 777], 8, -1, 0.03, 4, 128),       # GQA 8, two sequences
    (4, 2, [3000], 16, 200, 0.0, 2, 32),                 # GQA 2, 16 channels
    (32, 8, [131072 + 5], 8, -1, 0.03, 4, 128),          # the 128K Llama-3.1-8B shape
])
def test_group_selection_matches_oracle(Hq, Hkv, lengths, n_crit, k, ratio, ns, w):
    require_gpu()
    B, G = len(lengths), Hq // Hkv
    seed = synth.mix(synth.BASE_SEED + 1, 600, Hq, sum(lengths))
    KV = [synth.kv_rows(T, Hkv, synth.mix(seed, b)) for b, T in enumerate(lengths)]
    n_pages = sum(math.ceil(T / 16) for T in lengths) + 2
    alloc = kvq.Allocator(n_pages, seed=seed % 991 + 1)
    batch, _ = paged_batch(lengths, alloc)
    cache = kvq.LayerCache(Hq, Hkv, 16, n_pages, B, t_cap=(max(lengths) + 7) // 8 * 8)
    for b, T in enumerate(lengths):
        kvq.kv_quant_pack(cache, batch, b, 0, T, KV[b][0].cuda(), KV[b][1].cuda())
    q = synth.queries((B, Hq, 128), synth.mix(seed, 1))
    stride = (max(lengths) + 7) // 8 * 8
    sc = torch.full((B, Hkv, stride), float("nan"), device="cuda")
    crit = torch.full((B, Hkv, n_crit), -1, dtype=torch.int32, device="cuda")
    kvq.kv_group_critical_score(cache, batch, q.cuda(), n_crit, crit, sc)
    cap = max(O.topk_count(T, k if k >= 0 else O.ratio_k(T, ratio), ns, w) for T in lengths)
    sel = torch.full((B, Hkv, cap), -1, dtype=torch.int32, device="cuda")
    cnt = torch.zeros((B, Hkv), dtype=torch.int32, device="cuda")
    wt = ws(kvq.kv_topk_select_ws())
    kvq.kv_topk_select(batch, Hkv, sc, k, ratio, ns, w, sel, cnt, wt)
    out = torch.full((B, Hq, 128), float("nan"), device="cuda")
    wa = ws(kvq.kv_sparse_attn_ws(cache, batch, cap))
    kvq.kv_sparse_attn(cache, batch, q.cuda(), sel, cnt, 1, out, None, wa)
    for x in (wt, wa):
        kvq.kvq_check(x)
    sc_np, cr_np, sel_np, cnt_np, o = (x.cpu().numpy() for x in (sc, crit, sel, cnt, out))
    for b, T in enumerate(lengths):
        K, V = KV[b][0].numpy(), KV[b][1].numpy()
        kk = k if k >= 0 else O.ratio_k(T, ratio)
        for g in range(Hkv):
            qg = q[b, g * G:(g + 1) * G].numpy()
            C = O.group_critical_channels(qg, O.key_absmax(K[:, g]), n_crit)
            assert cr_np[b, g].tolist() == C.tolist(), (b, g)
            a = O.group_critical_scores(qg, K[:, g], C)
            assert np.array_equal(sc_np[b, g, :T].view(np.uint32), a.view(np.uint32)), (b, g)
            ids = O.topk_select(a, kk, ns, w)
            assert cnt_np[b, g] == len(ids) and sel_np[b, g, :len(ids)].tolist() == ids.tolist(), (b, g)
            for j in range(G):
                ref, _ = O.sparse_attn(qg[j], K[:, g], V[:, g], ids)
                assert attn_err(o[b, g * G + j], ref) <= ATTN_TOL, (b, g, j)
