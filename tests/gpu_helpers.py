"""Helpers for the GPU parity tests: library set-up, paged batches built with
the library's host allocator, and the normwise attention error metric."""
import math

import numpy as np
import pytest
import torch

from compressed_kv_cache_quant_gb300 import kvq
from compressed_kv_cache_quant_gb300.build import build

ATTN_TOL = 2e-3   # max |o - o_ref| / max |o_ref| per (sequence, head), fp32 accumulation


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()
    kvq.lib()


def paged_batch(capacities, allocator, lengths=None, shared_prefix_pages=None, share_with=None):
    """Block table with pages from `allocator` for sequences of the given token
    capacities.  shared_prefix_pages: number of leading pages that sequences in
    `share_with` take from sequence share_with[0] (reference counted)."""
    B = len(capacities)
    max_blocks = max(1, max(math.ceil(c / 16) for c in capacities))
    bt = np.full((B, max_blocks), -1, dtype=np.int32)
    for b, cap in enumerate(capacities):
        n = math.ceil(cap / 16)
        start = 0
        if shared_prefix_pages and share_with and b in share_with[1:]:
            src = share_with[0]
            for j in range(shared_prefix_pages):
                bt[b, j] = bt[src, j]
                allocator.ref(int(bt[src, j]))
            start = shared_prefix_pages
        ids = allocator.alloc(n - start)
        bt[b, start:n] = ids
    lens = np.array(lengths if lengths is not None else capacities, dtype=np.int32)
    max_len = int(max(capacities))
    batch = kvq.Batch(torch.from_numpy(bt).cuda(), torch.from_numpy(lens).cuda(), max_len)
    return batch, bt


def attn_err(o, ref):
    o = np.asarray(o, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(o - ref)) / den) if den > 0 else float(np.max(np.abs(o)))


def ws(nbytes):
    return kvq.Workspace(nbytes)
