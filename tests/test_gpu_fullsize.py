"""GPU parity at full size on the code paths the decode-step benchmark and the
serving-batch row run, through the C ABI, against the oracle.

* The sparse layer of the 128K Llama-3.1-8B-shaped step exactly as the
  benchmark calls it (no score copy, no selection output): every CTA attends
  its kept rows from the one-pass list; all 32 heads against the oracle's
  critical scores, top-K and exact attention.  A second case keeps about
  1000 rows per CTA, next to the list capacity, so that some CTAs compact; a
  third runs 200000 tokens.
* Layer 0 of the same step (1-bit K and V, groups of 64) at 131072 + 60
  prompt tokens plus 8 appended ones (a 64-token group completes during the
  appends): every warp of a CTA walks several groups through its double
  buffer (more than 16 groups per split).
* The INT4 serving batch at its stated shape: 16 sequences with lengths
  U[4096, 32768], 32 heads MHA, K 4-bit g64, V 4-bit G32, sequences 0-7
  sharing a 2048-token prefix (128 shared pages); the fixed 32-group split.

Sources: TailorKV §2.2, §2.3, §5.1; on-device article §3.1, §3.2;
KV-cache survey §一.1-§一.2, §三.1; meeting article §3.2."""
import math

import numpy as np
import pytest
import torch

from compressed_kv_cache_quant_gb300 import kvq, synth
from oracle import kvq_oracle as O
from gpu_helpers import ATTN_TOL, attn_err, paged_batch, require_gpu, ws
from kvq_format import k_row_codes, v_page_codes

pytestmark = pytest.mark.gpu

HQ, HKV = 32, 8


def _sparse_layer(T, seed):
    """An fp16 layer holding T - 1 prompt tokens of a 32 q / 8 kv head cache; the T-th
    token is handed to the decode call."""
    K, V = synth.kv_rows(T, HKV, seed)
    n_pages = math.ceil(T / 16) + 2
    alloc = kvq.Allocator(n_pages, seed=seed % 997 + 1)
    batch, bt = paged_batch([T], alloc, lengths=[T - 1])
    cache = kvq.LayerCache(HQ, HKV, 16, n_pages, 1, t_cap=(T + 7) // 8 * 8)
    kvq.kv_quant_pack(cache, batch, 0, 0, T - 1, K[:T - 1].cuda(), V[:T - 1].cuda())
    kvq.kvq_seq_lens_add(batch.seq_lens, 1)
    return K, V, cache, batch, bt, alloc


@pytest.mark.parametrize("T,k_fixed,ratio", [
    (131072 + 5, -1, 0.03),     # the benchmark's selection: K = floor(0.03 T), four CTAs per head
    (131072 + 5, 7900, 0.0),    # ~1000 kept rows per CTA, next to the list capacity (1024)
    (200000, -1, 0.03),         # a longer context: ~750 kept rows per CTA
])
def test_sparse_layer_bench_path_long(T, k_fixed, ratio):
    require_gpu()
    n_crit, ns, w = 8, 4, 128
    seed = synth.mix(synth.BASE_SEED + 1, 300, k_fixed, T)
    K, V, cache, batch, bt, _ = _sparse_layer(T, seed)
    q = synth.queries((1, HQ, 128), synth.mix(seed, 1))
    out = torch.full((1, HQ, 128), float("nan"), device="cuda")
    wk = ws(kvq.kv_sparse_layer_decode_ws())
    kvq.kv_sparse_layer_decode(cache, batch, K[T - 1][None].cuda(), V[T - 1][None].cuda(), q.cuda(), n_crit,
                               k_fixed, ratio, ns, w, out, wk)
    kvq.kvq_check(wk)
    listed, compacted, radix, _ = kvq.kvq_read_path_counters(wk)
    assert listed + compacted == HQ * 8 and radix == 0   # one cluster of 8 CTAs per q head
    if k_fixed < 0:
        assert compacted == 0         # every CTA attends its kept rows from the one-pass list
    else:
        assert listed > 0             # the CTAs whose kept rows fit the list; the others compact in order
    o = out.cpu().numpy()
    Kn, Vn = K.numpy(), V.numpy()
    kk = k_fixed if k_fixed >= 0 else O.ratio_k(T, ratio)
    for g in range(HKV):
        am = O.key_absmax(Kn[:, g])
        for h in range(g * HQ // HKV, (g + 1) * HQ // HKV):
            C = O.critical_channels(q[0, h].numpy(), am, n_crit)
            ids = O.topk_select(O.critical_scores(q[0, h].numpy(), Kn[:, g], C), kk, ns, w)
            ref, _ = O.sparse_attn(q[0, h].numpy(), Kn[:, g], Vn[:, g], ids)
            e = attn_err(o[0, h], ref)
            assert e <= ATTN_TOL, (h, e)
    # the append half of the step: the newest row is in the pages and the channel-major copy
    p = T - 1
    for g in range(HKV):
        assert np.array_equal(cache.k16[bt[0, p // 16], g, p % 16].cpu().numpy(), Kn[p, g])
        assert np.array_equal(cache.v16[bt[0, p // 16], g, p % 16].cpu().numpy(), Vn[p, g])
        assert np.array_equal(cache.kT[0, g, :, p].cpu().numpy(), Kn[p, g])


def _group_codes(cache_np, bt_row, g, h, bits):
    """Codes and (scale, zero) of 64-token group g of kv head h (pages 4g .. 4g + 3)."""
    pages = [int(bt_row[4 * g + j]) for j in range(4)]
    kc = np.concatenate([cache_np["k_codes"][p, h] for p in pages])            # [64][16 bits]
    vc = np.concatenate([v_page_codes(cache_np["v_codes"][p, h], bits) for p in pages])
    vsz = np.concatenate([cache_np["v_sz"][p, h] for p in pages])              # [64][d/G][2]
    return k_row_codes(kc, bits), cache_np["k_sz"][pages[0], h], vc, vsz


def test_quant_layer0_128k_append_and_attention():
    """Layer 0 of the 128K step: 1-bit K (per channel, g64) and V (per token, G64);
    131132 prompt tokens, then 8 appends: the 4th completes group 2048, the last
    four stay in the fp16 tail."""
    require_gpu()
    bits, G, T0, n_app = 1, 64, 131072 + 60, 8
    T = T0 + n_app
    seed = synth.mix(synth.BASE_SEED + 1, 301)
    K, V = synth.kv_rows(T, HKV, seed)
    n_pages = math.ceil(T / 16) + 2
    alloc = kvq.Allocator(n_pages, seed=13)
    batch, bt = paged_batch([T], alloc, lengths=[T0])
    cache = kvq.LayerCache(HQ, HKV, bits, n_pages, 1, v_group_dims=G)
    kvq.kv_quant_pack(cache, batch, 0, 0, T0, K[:T0].cuda(), V[:T0].cuda())
    wa = ws(kvq.kv_page_append_ws())
    for i in range(n_app):
        kvq.kvq_seq_lens_add(batch.seq_lens, 1)
        kvq.kv_page_append(cache, batch, K[T0 + i][None].cuda(), V[T0 + i][None].cuda(), wa)
    kvq.kvq_check(wa)
    n_splits, cps = kvq.kv_decode_attn_quant_plan(cache, batch)
    assert cps > 16, (n_splits, cps)      # 16 warps per CTA: every warp takes several groups
    q = synth.queries((1, HQ, 128), synth.mix(seed, 2))
    out = torch.full((1, HQ, 128), float("nan"), device="cuda")
    wq = ws(kvq.kv_decode_attn_quant_ws(cache, batch))
    kvq.kv_decode_attn_quant(cache, batch, q.cuda(), out, wq)
    kvq.kvq_check(wq)
    o = out.cpu().numpy()
    Kn, Vn = K.numpy(), V.numpy()
    pk = [O.pack_k(Kn[:, g], bits) for g in range(HKV)]
    pv = [O.pack_v(Vn[:, g], bits, G) for g in range(HKV)]
    ref = O.decode_attn_quant(q[0].numpy(), pk, pv)
    for h in range(HQ):
        e = attn_err(o[0, h], ref[h])
        assert e <= ATTN_TOL, (h, e)
    # the group the appends completed, and the last group of the prompt, bit for bit
    cnp = {k: getattr(cache, k).cpu().numpy() for k in ("k_codes", "v_codes", "k_sz", "v_sz", "k_tail")}
    for grp in (2047, 2048):
        for g in (0, 5):
            kc, ksz, vc, vsz = _group_codes(cnp, bt[0], grp, g, bits)
            t = slice(64 * grp, 64 * grp + 64)
            assert np.array_equal(kc, pk[g]["codes"][t])
            assert np.array_equal(ksz[:, 0].view(np.uint16), pk[g]["scale16"][grp].view(np.uint16))
            assert np.array_equal(ksz[:, 1].view(np.uint16), pk[g]["zero16"][grp].view(np.uint16))
            assert np.array_equal(vc, pv[g]["codes"][t])
            assert np.array_equal(vsz[..., 0].view(np.uint16), pv[g]["scale16"][t].view(np.uint16))
    for g in range(HKV):
        nt = T - pk[g]["n_packed"]
        assert nt == T % 64 == 4
        assert np.array_equal(cnp["k_tail"][0, g, :nt].view(np.uint16), pk[g]["tail"].view(np.uint16))


def test_int4_serving_batch_stated_shape():
    """16 sequences, T ~ U[4096, 32768], 32 heads MHA, K 4-bit g64, V 4-bit G32,
    sequences 0-7 sharing the first 128 pages (2048 tokens) of sequence 0; the
    split takes a fixed 32 groups.  Two heads of every sequence are checked."""
    require_gpu()
    bits, G, H, B, pre = 4, 32, 32, 16, 2048
    seed = synth.BASE_SEED + 2
    lens = [int(x) for x in synth.lengths_uniform(B, 4096, 32768, seed)]
    n_pages = sum(math.ceil(T / 16) for T in lens) + 4
    alloc = kvq.Allocator(n_pages, seed=seed % 1000 + 7)
    share = list(range(8))
    batch, bt = paged_batch(lens, alloc, shared_prefix_pages=pre // 16, share_with=share)
    assert all(alloc.refcount(int(bt[0, j])) == 8 for j in (0, 127))
    cache = kvq.LayerCache(H, H, bits, n_pages, B, v_group_dims=G)
    heads = {b: [(3 * b) % H, (3 * b + 17) % H] for b in range(B)}
    host = {}
    prefix = None
    for b, T in enumerate(lens):
        K, V = synth.kv_rows(T, H, synth.mix(seed, 10 + b), device="cuda")
        if b == 0:
            prefix = (K[:pre].clone(), V[:pre].clone())
        elif b in share:
            K[:pre], V[:pre] = prefix
        t0 = pre if (b in share and b > 0) else 0
        kvq.kv_quant_pack(cache, batch, b, t0, T - t0, K[t0:], V[t0:])
        host[b] = (K[:, heads[b]].cpu().numpy(), V[:, heads[b]].cpu().numpy())
        del K, V
    torch.cuda.synchronize()
    n_splits, cps = kvq.kv_decode_attn_quant_plan(cache, batch)
    assert cps == 32 and n_splits == math.ceil(max(lens) / 64 / 32), (n_splits, cps)
    q = synth.queries((B, H, 128), synth.mix(seed, 99))
    out = torch.full((B, H, 128), float("nan"), device="cuda")
    wq = ws(kvq.kv_decode_attn_quant_ws(cache, batch))
    kvq.kv_decode_attn_quant(cache, batch, q.cuda(), out, wq)
    kvq.kvq_check(wq)
    o = out.cpu().numpy()
    for b, T in enumerate(lens):
        Kh, Vh = host[b]
        for j, h in enumerate(heads[b]):
            pk, pv = O.pack_k(Kh[:, j], bits), O.pack_v(Vh[:, j], bits, G)
            ref = O.decode_attn_quant(q[b, h:h + 1].numpy(), [pk], [pv])
            e = attn_err(o[b, h], ref[0])
            assert e <= ATTN_TOL, (b, h, T, e)


def test_pack_qwen14b_layer_40_heads():
    """One Qwen-1.5-14B-shaped layer packed to 1 bit in one call: 40 kv heads x
    131072 tokens, K per channel g64, V per token G64; three heads bit for bit
    against the oracle (codes, scales, zeros)."""
    require_gpu()
    bits, G, H, T = 1, 64, 40, 131072
    K, V = synth.kv_rows(T, H, synth.mix(synth.BASE_SEED + 5, 302), device="cuda")
    n_pages = T // 16
    alloc = kvq.Allocator(n_pages, seed=17)
    batch, bt = paged_batch([T], alloc)
    cache = kvq.LayerCache(H, H, bits, n_pages, 1, v_group_dims=G)
    kvq.kv_quant_pack(cache, batch, 0, 0, T, K, V)
    torch.cuda.synchronize()
    heads = (0, 17, 39)
    Kh, Vh = K[:, heads].cpu().numpy(), V[:, heads].cpu().numpy()
    del K, V
    for j, h in enumerate(heads):
        pk, pv = O.pack_k(Kh[:, j], bits), O.pack_v(Vh[:, j], bits, G)
        kc = k_row_codes(cache.k_codes[:, h].cpu().numpy()[bt[0]].reshape(T, -1), bits)
        assert np.array_equal(kc, pk["codes"]), h
        ksz = cache.k_sz[:, h].cpu().numpy()[bt[0][0::4]]                 # [groups][d][2]
        assert np.array_equal(ksz[..., 0].view(np.uint16), pk["scale16"].view(np.uint16)), h
        assert np.array_equal(ksz[..., 1].view(np.uint16), pk["zero16"].view(np.uint16)), h
        vc = v_page_codes(cache.v_codes[:, h].cpu().numpy()[bt[0]], bits).reshape(T, 128)
        assert np.array_equal(vc, pv["codes"]), h
        vsz = cache.v_sz[:, h].cpu().numpy()[bt[0]].reshape(T, -1, 2)
        assert np.array_equal(vsz[..., 0].view(np.uint16), pv["scale16"].view(np.uint16)), h
        assert np.array_equal(vsz[..., 1].view(np.uint16), pv["zero16"].view(np.uint16)), h
