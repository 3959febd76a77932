"""GPU parity of a3 kv_decode_attn_quant against the oracle (fp64) on the same
seeded caches: normwise error <= 2e-3 per (sequence, head); ragged tails,
empty and one-token sequences, GQA 4 and MHA, shared-prefix pages."""
import math

import numpy as np
import pytest
import torch

from compressed_kv_cache_quant_gb300 import kvq, synth
from oracle import kvq_oracle as O
from gpu_helpers import ATTN_TOL, attn_err, paged_batch, require_gpu, ws

pytestmark = pytest.mark.gpu


def _run(bits, G, Hq, Hkv, lengths, seed, share=None):
    B = len(lengths)
    KV = [synth.kv_rows(max(T, 1), Hkv, synth.mix(seed, b)) for b, T in enumerate(lengths)]
    if share:   # sequences share[1:] reuse the first `pre` tokens of share[0]
        pre, members = share
        for b in members[1:]:
            KV[b] = (torch.cat([KV[members[0]][0][:pre], KV[b][0][pre:]]),
                     torch.cat([KV[members[0]][1][:pre], KV[b][1][pre:]]))
    n_pages = sum(math.ceil(max(T, 1) / 16) for T in lengths) + 4
    alloc = kvq.Allocator(n_pages, seed=seed % 1000 + 1)
    if share:
        batch, bt = paged_batch([max(T, 1) for T in lengths], alloc, lengths=lengths,
                                shared_prefix_pages=share[0] // 16, share_with=share[1])
    else:
        batch, bt = paged_batch([max(T, 1) for T in lengths], alloc, lengths=lengths)
    cache = kvq.LayerCache(Hq, Hkv, bits, n_pages, B, v_group_dims=G)
    for b, T in enumerate(lengths):
        t0 = share[0] if (share and b in share[1][1:]) else 0
        if T > t0:
            kvq.kv_quant_pack(cache, batch, b, t0, T - t0, KV[b][0][t0:T].cuda(), KV[b][1][t0:T].cuda())
    q = synth.queries((B, Hq, 128), synth.mix(seed, 99))
    out = torch.full((B, Hq, 128), float("nan"), device="cuda")
    w = ws(kvq.kv_decode_attn_quant_ws(cache, batch))
    kvq.kv_decode_attn_quant(cache, batch, q.cuda(), out, w)
    kvq.kvq_check(w)
    o = out.cpu().numpy()
    for b, T in enumerate(lengths):
        if T == 0:
            assert np.all(o[b] == 0)
            continue
        K, V = KV[b][0][:T].numpy(), KV[b][1][:T].numpy()
        pk = [O.pack_k(K[:, g], bits) for g in range(Hkv)]
        pv = [O.pack_v(V[:, g], bits, G) for g in range(Hkv)]
        ref = O.decode_attn_quant(q[b].numpy(), pk, pv)
        for h in range(Hq):
            e = attn_err(o[b, h], ref[h])
            assert e <= ATTN_TOL, (b, h, T, e)
    # a second call on the same workspace gives the same result (counters were reset)
    out2 = torch.empty_like(out)
    kvq.kv_decode_attn_quant(cache, batch, q.cuda(), out2, w)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_config_tiny_one_bit_gqa4():
    """Tiny single layer: 8 q / 2 kv heads, T=4096, K and V 1-bit, group 64."""
    require_gpu()
    _run(1, 64, 8, 2, [4096], synth.mix(synth.BASE_SEED + 0, 1))


@pytest.mark.parametrize("bits,G", [(1, 64), (2, 32), (4, 32), (8, 128)])
def test_ragged_lengths_in_one_batch(bits, G):
    require_gpu()
    _run(bits, G, 8, 2, [1, 63, 64, 65, 1000, 4096 + 37, 0], synth.mix(synth.BASE_SEED, 2, bits))


def test_mha_int4_shared_prefix():
    """INT4 (K g64, V g32) MHA batch; sequences 0..2 share a 256-token prefix."""
    require_gpu()
    lengths = [700, 1300, 257, 2100]
    _run(4, 32, 8, 8, lengths, synth.mix(synth.BASE_SEED + 2, 3), share=(256, [0, 1, 2]))


@pytest.mark.parametrize("gq,G", [(1, 64), (2, 64), (8, 64), (2, 32), (1, 128)])
def test_gqa_widths(gq, G):
    """Query heads per kv head against V groups per token: the value product gives each
    (head, V group) a column of its own when they fit (2 heads x 4 groups fill all eight)."""
    require_gpu()
    seed = synth.mix(synth.BASE_SEED, 4, gq) if G == 64 else synth.mix(synth.BASE_SEED, 4, gq, G)
    _run(2, G, 2 * gq, 2, [333, 900], seed)


def test_v_scale_beyond_fp16_range_is_flagged():
    """With the V scales in the value product's B operand as fp16(2^8 p vscale), a V group
    whose scale reaches 256 (1-bit codes of values up to about +-1000) is reported as a
    range error by the status word rather than giving an invalid output silently."""
    require_gpu()
    T, Hq, Hkv = 256, 8, 2
    K, V = synth.kv_rows(T, Hkv, synth.mix(synth.BASE_SEED, 5))
    V = (V.float() * 300.0).to(torch.float16)
    alloc = kvq.Allocator(T // 16 + 4, seed=5)
    batch, bt = paged_batch([T], alloc, lengths=[T])
    cache = kvq.LayerCache(Hq, Hkv, 1, T // 16 + 4, 1, v_group_dims=64)
    kvq.kv_quant_pack(cache, batch, 0, 0, T, K.cuda(), V.cuda())
    q = synth.queries((1, Hq, 128), synth.mix(synth.BASE_SEED, 6))
    out = torch.empty((1, Hq, 128), device="cuda")
    w = ws(kvq.kv_decode_attn_quant_ws(cache, batch))
    kvq.kv_decode_attn_quant(cache, batch, q.cuda(), out, w)
    with pytest.raises(kvq.KvqError, match="fp16 range"):
        kvq.kvq_check(w)
