"""GPU parity of the FP8 E4M3 layer (meeting article, section 6 item 2): the
pack and the append store every fp16 value as its E4M3 byte (bit-exact against
the oracle, every fp16 pattern), and decode attention over the E4M3 cache -- bulk
asynchronous copies into shared memory, tensor-core products -- is within 2e-3
of the oracle's exact attention over the E4M3 values."""
import math

import numpy as np
import pytest
import torch

from compressed_kv_cache_quant_gb300 import kvq, synth
from oracle import kvq_oracle as O
from gpu_helpers import ATTN_TOL, attn_err, paged_batch, require_gpu, ws

pytestmark = pytest.mark.gpu
E4M3 = kvq.BITS_E4M3


def _rows(cache, bt_row, T, h):
    """Logical [T][d] K and V bytes of kv head h of one sequence."""
    kc, vc = cache.k_codes.cpu().numpy(), cache.v_codes.cpu().numpy()
    idx = [int(bt_row[t // 16]) for t in range(T)]
    return (np.stack([kc[idx[t], h, t % 16] for t in range(T)]), np.stack([vc[idx[t], h, t % 16] for t in range(T)]))


def test_pack_every_fp16_value_and_append():
    require_gpu()
    H, T0 = 1, 512
    allv = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.float16).reshape(T0, H, 128)
    K = allv.clone()
    V = allv.flip(0).clone()
    extra = synth.kv_rows(3, H, 77)
    n_pages = math.ceil((T0 + 3) / 16)
    alloc = kvq.Allocator(n_pages, seed=3)
    batch, bt = paged_batch([T0 + 3], alloc, lengths=[T0])
    cache = kvq.LayerCache(4, H, E4M3, n_pages, 1)
    kvq.kv_quant_pack(cache, batch, 0, 0, T0, K.cuda(), V.cuda())
    w = ws(kvq.kv_page_append_ws())
    for i in range(3):
        kvq.kvq_seq_lens_add(batch.seq_lens, 1)
        kvq.kv_page_append(cache, batch, extra[0][i][None].cuda(), extra[1][i][None].cuda(), w)
    kvq.kvq_check(w)
    kb, vb = _rows(cache, bt[0], T0 + 3, 0)
    Kall = torch.cat([K, extra[0]]).numpy()[:, 0]
    Vall = torch.cat([V, extra[1]]).numpy()[:, 0]
    for got, x in ((kb, Kall), (vb, Vall)):
        want = O.fp8_e4m3_encode(x)
        nan = np.isnan(x.astype(np.float32))
        assert np.array_equal(got[~nan], want[~nan])
        assert np.all((got[nan] & 0x7F) == 0x7F)


def _attn_case(Hq, Hkv, lengths, seed):
    B = len(lengths)
    KV = [synth.kv_rows(max(T, 1), Hkv, synth.mix(seed, b)) for b, T in enumerate(lengths)]
    n_pages = sum(math.ceil(max(T, 1) / 16) for T in lengths) + 2
    alloc = kvq.Allocator(n_pages, seed=seed % 1000 + 1)
    batch, _ = paged_batch([max(T, 1) for T in lengths], alloc, lengths=lengths)
    cache = kvq.LayerCache(Hq, Hkv, E4M3, n_pages, B)
    for b, T in enumerate(lengths):
        if T:
            kvq.kv_quant_pack(cache, batch, b, 0, T, KV[b][0][:T].cuda(), KV[b][1][:T].cuda())
    q = synth.queries((B, Hq, 128), synth.mix(seed, 9))
    out = torch.full((B, Hq, 128), float("nan"), device="cuda")
    wq = ws(kvq.kv_decode_attn_quant_ws(cache, batch))
    kvq.kv_decode_attn_quant(cache, batch, q.cuda(), out, wq)
    kvq.kvq_check(wq)
    out2 = torch.empty_like(out)
    kvq.kv_decode_attn_quant(cache, batch, q.cuda(), out2, wq)   # the counters were reset
    torch.cuda.synchronize()
    assert torch.equal(out, out2)
    return KV, q, out.cpu().numpy(), cache, batch


@pytest.mark.parametrize("Hq,Hkv,lengths", [
    (8, 2, [4096]),
    (8, 2, [1, 15, 16, 17, 31, 32, 33, 1000, 4096 + 37, 0]),
    (8, 8, [700, 2100]),
    (16, 2, [333, 5000]),
    (4, 2, [64, 129]),
])
def test_decode_attention_matches_oracle(Hq, Hkv, lengths):
    require_gpu()
    KV, q, o, _, _ = _attn_case(Hq, Hkv, lengths, synth.mix(synth.BASE_SEED, 700, Hq, Hkv, len(lengths)))
    for b, T in enumerate(lengths):
        if T == 0:
            assert np.all(o[b] == 0)
            continue
        for h in range(Hq):
            g = O.kv_head_of(h, Hq, Hkv)
            ref, _ = O.fp8_attention(q[b, h].numpy(), KV[b][0][:T, g].numpy(), KV[b][1][:T, g].numpy())
            e = attn_err(o[b, h], ref)
            assert e <= ATTN_TOL, (b, h, T, e)


def test_decode_attention_128k():
    """32 q / 8 kv heads over 131072 + 37 tokens: each warp walks its steps through the
    two stages many times."""
    require_gpu()
    T = 131072 + 37
    KV, q, o, cache, batch = _attn_case(32, 8, [T], synth.mix(synth.BASE_SEED, 701))
    n_splits, cps = kvq.kv_decode_attn_quant_plan(cache, batch)
    assert 2 * cps > 12 * 4, (n_splits, cps)       # more than four steps per warp
    for h in (0, 5, 13, 22, 31):
        g = O.kv_head_of(h, 32, 8)
        ref, _ = O.fp8_attention(q[0, h].numpy(), KV[0][0][:, g].numpy(), KV[0][1][:, g].numpy())
        assert attn_err(o[0, h], ref) <= ATTN_TOL, h


def test_bounded_wait_gives_up_with_a_status():
    """The E4M3 kernel's wait for its bulk copies is bounded: run on a barrier that nothing
    completes, it gives up, the workspace status word says so, and the context stays usable."""
    import time
    require_gpu()
    w = ws(256)
    t0 = time.time()
    kvq.kvq_selftest_bounded_wait(w)
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_check(w)
    assert e.value.code == -6 and "bounded wait" in str(e.value)
    assert time.time() - t0 < 60
    kvq.kvq_check(w)                       # the status word was cleared
    x = torch.arange(8, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 28.0          # later work runs normally
