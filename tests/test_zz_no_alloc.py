"""The allocation-free decode attention (kv_decode_attn_quant_noalloc) against
the workspace version, through the C ABI.

Some callers cannot give the library device memory (a plugin whose framework
owns every allocation, a decode loop that must not enter the CUDA allocator);
they call the variant that keeps its split-K scratch in an array built into
the library.  This file is collected last on purpose: the variant shares one
array across all calls, and the test must hold both in a fresh process and
after every other test has run."""
import math

import numpy as np
import pytest
import torch

from compressed_kv_cache_quant_gb300 import _abi, kvq, synth
from gpu_helpers import ATTN_TOL, attn_err, paged_batch, require_gpu, ws

pytestmark = pytest.mark.gpu


def _layer(bits, G, Hq, Hkv, lengths, seed):
    B = len(lengths)
    KV = [synth.kv_rows(T, Hkv, synth.mix(seed, b)) for b, T in enumerate(lengths)]
    n_pages = sum(math.ceil(T / 16) for T in lengths) + 2
    alloc = kvq.Allocator(n_pages, seed=31)
    batch, _ = paged_batch(lengths, alloc)
    cache = kvq.LayerCache(Hq, Hkv, bits, n_pages, B, v_group_dims=G)
    for b, T in enumerate(lengths):
        kvq.kv_quant_pack(cache, batch, b, 0, T, KV[b][0].cuda(), KV[b][1].cuda())
    return cache, batch


@pytest.mark.parametrize("bits,G,Hq,Hkv,lengths", [(1, 64, 8, 2, [4096]), (4, 32, 8, 8, [700, 1300, 33])])
def test_noalloc_matches_workspace_version_twice(bits, G, Hq, Hkv, lengths):
    require_gpu()
    cache, batch = _layer(bits, G, Hq, Hkv, lengths, synth.mix(synth.BASE_SEED, 900, bits))
    B = len(lengths)
    q = synth.queries((B, Hq, 128), synth.mix(synth.BASE_SEED, 901, bits)).cuda()
    ref = torch.empty((B, Hq, 128), device="cuda")
    kvq.kv_decode_attn_quant(cache, batch, q, ref, ws(kvq.kv_decode_attn_quant_ws(cache, batch)))
    assert kvq.kv_decode_attn_quant_ws(cache, batch) <= kvq.kv_decode_attn_quant_noalloc_max_scratch()
    for _ in range(2):   # the second call reuses the array the first one left behind
        out = torch.full((B, Hq, 128), float("nan"), device="cuda")
        kvq.kv_decode_attn_quant_noalloc(cache, batch, q, out)
        torch.cuda.synchronize()
        o, r = out.cpu().numpy(), ref.cpu().numpy()
        for b in range(B):
            for h in range(Hq):
                assert attn_err(o[b, h], r[b, h]) <= ATTN_TOL


def test_noalloc_rejects_batches_beyond_the_array():
    require_gpu()
    cache, batch = _layer(1, 64, 8, 8, [64], 5)
    huge = kvq.Batch(batch.block_table, batch.seq_lens, batch.max_len)
    huge.c.batch = 1
    # pretend a batch of 4096 sequences: the scratch it needs exceeds 8 MiB
    big = _abi.Seqs(huge.c.block_table, huge.c.seq_lens, 4096, huge.c.max_blocks, huge.c.max_len, 0)
    cache.c.max_seqs = 4096
    need = kvq.lib().kv_decode_attn_quant_ws(kvq._ref(cache.layout), kvq._ref(big))
    assert need > kvq.kv_decode_attn_quant_noalloc_max_scratch()
    st = kvq.lib().kv_decode_attn_quant_noalloc(kvq._ref(cache.layout), kvq._ref(cache), kvq._ref(big),
                                                None, None, None)
    assert st == _abi.KVQ_ERR_NO_SPACE
    assert "scratch" in _abi.last_error()


def test_noalloc_compact_plan_when_the_default_does_not_fit():
    """A batch whose default split needs more scratch than the built-in array (16
    sequences of 32 MHA heads, one of them 65536 tokens long): the allocation-free
    call plans fewer, longer splits, and twice in a row still gives the workspace
    version's result."""
    require_gpu()
    lengths = [65536] + [100 + 7 * i for i in range(15)]
    cache, batch = _layer(4, 32, 32, 32, lengths, synth.mix(synth.BASE_SEED, 902))
    assert kvq.kv_decode_attn_quant_ws(cache, batch) > kvq.kv_decode_attn_quant_noalloc_max_scratch()
    plan_ws = kvq.kv_decode_attn_quant_plan(cache, batch)
    plan_na = kvq.kv_decode_attn_quant_plan(cache, batch, noalloc=True)
    assert plan_na[0] < plan_ws[0], (plan_na, plan_ws)
    B, Hq = len(lengths), 32
    q = synth.queries((B, Hq, 128), synth.mix(synth.BASE_SEED, 903)).cuda()
    ref = torch.empty((B, Hq, 128), device="cuda")
    kvq.kv_decode_attn_quant(cache, batch, q, ref, ws(kvq.kv_decode_attn_quant_ws(cache, batch)))
    r = ref.cpu().numpy()
    for _ in range(2):
        out = torch.full((B, Hq, 128), float("nan"), device="cuda")
        kvq.kv_decode_attn_quant_noalloc(cache, batch, q, out)
        torch.cuda.synchronize()
        o = out.cpu().numpy()
        for b in range(B):
            for h in range(Hq):
                assert attn_err(o[b, h], r[b, h]) <= ATTN_TOL, (b, h)
