"""GPU parity of the mixed layer (TailorKV section 6: the layer-level strategy
carried down to heads): kv heads classified dense attend every token, the others
take critical scores + top-K + attention, dispatched on the device by each head's
class (the cluster launch for the sparse heads and the appends, then the dense kv
heads' GQA-shared attention); the optional selection copy (every token for a
dense head, the top-K set for a sparse one); and the classification itself from
GPU dense-preference scores.
Sources: TailorKV §2.1, §2.3, §5.1, §6; KV-cache survey §三.1; meeting article §3.2."""
import math

import numpy as np
import pytest
import torch

from compressed_kv_cache_quant_gb300 import kvq, synth
from oracle import kvq_oracle as O
from gpu_helpers import ATTN_TOL, attn_err, paged_batch, require_gpu, ws

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("Hq,Hkv,T,dense,with_sel", [
    (8, 2, 4096 + 5, [1, 0], False),
    (8, 2, 3000, [0, 1], True),
    (32, 8, 131072 + 5, [1, 0, 0, 0, 0, 0, 1, 0], False),
    (32, 8, 70000, [0, 1, 1, 0, 0, 0, 0, 1], True),
    (8, 8, 2000, [1, 0, 1, 0, 0, 0, 0, 1], False),
])
def test_mixed_layer_matches_oracle(Hq, Hkv, T, dense, with_sel):
    require_gpu()
    G = Hq // Hkv
    seed = synth.mix(synth.BASE_SEED + 1, 900, Hq, T)
    K, V = synth.kv_rows(T, Hkv, seed)
    n_pages = math.ceil(T / 16) + 2
    alloc = kvq.Allocator(n_pages, seed=5)
    batch, bt = paged_batch([T], alloc, lengths=[T - 1])
    cache = kvq.LayerCache(Hq, Hkv, 16, n_pages, 1, t_cap=(T + 7) // 8 * 8)
    kvq.kv_quant_pack(cache, batch, 0, 0, T - 1, K[:T - 1].cuda(), V[:T - 1].cuda())
    kvq.kvq_seq_lens_add(batch.seq_lens, 1)
    q = synth.queries((1, Hq, 128), synth.mix(seed, 1))
    out = torch.full((1, Hq, 128), float("nan"), device="cuda")
    dn = torch.tensor([dense], dtype=torch.int32, device="cuda")
    wk = ws(kvq.kv_mixed_layer_decode_ws(cache, batch))
    sel = torch.full((1, Hq, T), -7, dtype=torch.int32, device="cuda") if with_sel else None
    cnt = torch.full((1, Hq), -7, dtype=torch.int32, device="cuda") if with_sel else None
    kvq.kv_mixed_layer_decode(cache, batch, K[T - 1][None].cuda(), V[T - 1][None].cuda(), q.cuda(), 8, -1, 0.03, 4,
                              128, dn, out, wk, sel=sel, sel_count=cnt)
    kvq.kvq_check(wk)
    o, Kn, Vn = out.cpu().numpy(), K.numpy(), V.numpy()
    heads = range(Hq) if Hq <= 8 else [0, 1, 5, 24, 25, 31]
    for h in heads:
        g = h // G
        if dense[g]:
            ids = np.arange(T)
        else:
            C = O.critical_channels(q[0, h].numpy(), O.key_absmax(Kn[:, g]), 8)
            ids = O.topk_select(O.critical_scores(q[0, h].numpy(), Kn[:, g], C), O.ratio_k(T, 0.03), 4, 128)
        ref, _ = O.sparse_attn(q[0, h].numpy(), Kn[:, g], Vn[:, g], ids)
        assert attn_err(o[0, h], ref) <= ATTN_TOL, (h, dense[g])
        if with_sel:
            n = int(cnt[0, h])
            assert n == len(ids) and np.array_equal(sel[0, h, :n].cpu().numpy(), ids), (h, dense[g])
    # a second call on the same workspace (counters were left zeroed): the dense heads' outputs bit
    # for bit (fixed order of tiles, warps and splits); the sparse heads' kept rows are collected in
    # arrival order, so their fp32 sums may differ in the last bits
    out2 = torch.full_like(out, float("nan"))
    kvq.kv_mixed_layer_decode(cache, batch, K[T - 1][None].cuda(), V[T - 1][None].cuda(), q.cuda(), 8, -1, 0.03, 4,
                              128, dn, out2, wk)
    torch.cuda.synchronize()
    o2 = out2.cpu().numpy()
    for h in range(Hq):
        if dense[h // G]:
            assert np.array_equal(o2[0, h], o[0, h]), h
        else:
            assert np.allclose(o2[0, h], o[0, h], rtol=1e-5, atol=1e-6 * np.abs(o[0, h]).max()), h
    p = T - 1
    for g in range(Hkv):   # the newest token appended for dense and sparse kv heads alike
        assert np.array_equal(cache.k16[bt[0, p // 16], g, p % 16].cpu().numpy(), Kn[p, g])
        assert np.array_equal(cache.kT[0, g, :, p].cpu().numpy(), Kn[p, g])


def test_classification_from_gpu_scores():
    """Dense-preference scores on the GPU, then the per-kv-head classes: the same classes as
    the oracle's scores give (config 1's shape: 8 q / 2 kv heads, T = 4096, 32 recent queries,
    top-128, tau 0.2), one kv head's queries made dense (q = 0: uniform attention)."""
    require_gpu()
    Hq, Hkv, T, n_q, topk = 8, 2, 4096, 32, 128
    K, V = synth.kv_rows(T, Hkv, synth.mix(synth.BASE_SEED, 901))
    n_pages = T // 16
    alloc = kvq.Allocator(n_pages, seed=3)
    batch, _ = paged_batch([T], alloc)
    cache = kvq.LayerCache(Hq, Hkv, 16, n_pages, 1, t_cap=T)
    kvq.kv_quant_pack(cache, batch, 0, 0, T, K.cuda(), V.cuda())
    Q = synth.queries((1, Hq, n_q, 128), synth.mix(synth.BASE_SEED, 902)) * 4
    Q[0, :4] = 0                                    # kv head 0's queries: uniform attention, P near n_q
    P = torch.empty((1, Hq), device="cuda")
    wd = ws(kvq.kv_dense_pref_score_ws(cache, batch, n_q))
    kvq.kv_dense_pref_score(cache, batch, Q.cuda(), n_q, topk, P, wd)
    kvq.kvq_check(wd)
    Pg = P.cpu().numpy()[0]
    ref = [O.dense_pref_score(Q[0, h].numpy(), K[:, h // 4].numpy(), topk) for h in range(Hq)]
    want = [int(x) for x in O.classify_heads(ref, n_q, 0.2, Hkv)]
    got = kvq.kvq_classify_heads(Pg.tolist(), Hq, Hkv, n_q, 0.2)
    assert got == want and got[0] == 1
