"""Host-side checks of the C ABI (no GPU compute): the library loads, exports
every function include/kvq.h declares, validates arguments before launching
anything, and its host page allocator keeps free lists and reference counts."""
import ctypes
import os
import re

import pytest

from compressed_kv_cache_quant_gb300 import _abi, kvq
from compressed_kv_cache_quant_gb300.build import build

pytestmark = pytest.mark.cpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return kvq.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b((?:kv|kvq)_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_function(lib):
    names = header_functions()
    assert len(names) >= 28
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_abi.PROTOTYPES), set(names) ^ set(_abi.PROTOTYPES)
    assert lib.kvq_version() == _abi.ABI_VERSION


def test_validation_rejects_before_launch(lib):
    L = kvq.make_layout(8, 2, 1, 64)
    P = _abi.Pool()
    S = _abi.Seqs(None, None, 0, 0, 0, 0)
    by = ctypes.byref
    # NULL layout / unsupported geometry / bad group size
    assert lib.kv_decode_attn_quant(None, by(P), by(S), None, None, None, 0, None) == _abi.KVQ_ERR_INVALID_ARG
    bad = kvq.make_layout(8, 2, 3, 64)
    assert lib.kv_decode_attn_quant(by(bad), by(P), by(S), None, None, None, 0, None) == _abi.KVQ_ERR_UNSUPPORTED
    assert "bits" in _abi.last_error()
    bad = kvq.make_layout(8, 2, 4, 48)
    assert lib.kv_quant_pack(by(bad), by(P), by(S), 0, 0, 0, None, None, 0, None) == _abi.KVQ_ERR_UNSUPPORTED
    bad = kvq.make_layout(6, 4, 4, 64)
    assert lib.kv_sparse_attn(by(bad), by(P), by(S), None, None, 1, None, 0, None, None, None, 0, None) \
        == _abi.KVQ_ERR_INVALID_ARG
    # missing pool arrays
    assert lib.kv_decode_attn_quant(by(L), by(P), by(S), None, None, None, 0, None) == _abi.KVQ_ERR_INVALID_ARG
    # workspace too small / misaligned
    assert lib.kv_page_append(by(L), by(P), by(S), None, None, 256, 16, None) == _abi.KVQ_ERR_INVALID_ARG
    assert lib.kv_topk_select(by(S), 1, None, 0, 1, 0.0, 0, 0, None, 1, None, 8, 256, None) \
        == _abi.KVQ_ERR_INVALID_ARG
    # too-long context for the cluster top-k
    S2 = _abi.Seqs(None, None, 0, 100000, 8 * 49152 + 8, 0)
    assert lib.kv_topk_select(by(S2), 1, 1024, 8 * 49152 + 8, 1, 0.0, 0, 0, 1024, 1, 1024, 256, 256, None) \
        == _abi.KVQ_ERR_UNSUPPORTED
    # max_len beyond the block table
    S3 = _abi.Seqs(None, None, 0, 2, 33, 0)
    assert lib.kv_page_append(by(L), by(P), by(S3), None, None, 256, 256, None) == _abi.KVQ_ERR_INVALID_ARG


def test_block_select_validation(lib):
    """kv_block_select rejects bad arguments on the host, before any launch."""
    by = ctypes.byref
    S = _abi.Seqs(None, None, 0, 8, 100, 0)
    # block size, sink/window, ratio, capacity
    assert lib.kv_block_select(by(S), 1, 8, 128, -1, 0.03, 4, 64, 0, 8, 16, 8, None, 0, None) \
        == _abi.KVQ_ERR_INVALID_ARG
    assert "block_tokens" in _abi.last_error()
    assert lib.kv_block_select(by(S), 1, 8, 128, -1, 0.03, -1, 64, 64, 8, 16, 8, None, 0, None) \
        == _abi.KVQ_ERR_INVALID_ARG
    assert lib.kv_block_select(by(S), 1, 8, 128, -1, 1.5, 4, 64, 64, 8, 16, 8, None, 0, None) \
        == _abi.KVQ_ERR_INVALID_ARG
    assert lib.kv_block_select(by(S), 1, 8, 128, -1, 0.03, 4, 64, 64, 8, 0, 8, None, 0, None) \
        == _abi.KVQ_ERR_INVALID_ARG
    # score stride below max_len
    assert lib.kv_block_select(by(S), 1, 8, 64, -1, 0.03, 4, 64, 64, 8, 16, 8, None, 0, None) \
        == _abi.KVQ_ERR_INVALID_ARG
    # more blocks per row than the selection CTA holds
    S2 = _abi.Seqs(None, None, 0, 30000, 400000, 0)
    need = lib.kv_block_select_ws(by(S2), 1, 16)
    assert lib.kv_block_select(by(S2), 1, 8, 400000, -1, 0.03, 4, 64, 16, 8, 16, 8, None, need, None) \
        == _abi.KVQ_ERR_UNSUPPORTED
    # workspace too small
    assert lib.kv_block_select(by(S), 1, 8, 128, -1, 0.03, 4, 64, 64, 8, 16, 8, None, 16, None) \
        == _abi.KVQ_ERR_INVALID_ARG
    # sizes: importances of every row, 256-byte aligned; 0 for invalid arguments
    S3 = _abi.Seqs(None, None, 2, 8200, 131136, 0)
    n = lib.kv_block_select_ws(by(S3), 32, 64)
    assert n % 256 == 0 and n >= 256 + 2 * 32 * 2052 * 4
    assert lib.kv_block_select_ws(by(S3), 0, 64) == 0 and lib.kv_block_select_ws(by(S3), 32, 0) == 0


def test_workspace_sizes(lib):
    L = kvq.make_layout(32, 8, 1, 64)
    S = _abi.Seqs(None, None, 1, 8200, 131136, 0)
    n = lib.kv_decode_attn_quant_ws(ctypes.byref(L), ctypes.byref(S))
    assert n >= 256 and n % 256 == 0
    m = lib.kv_sparse_attn_ws(ctypes.byref(L), ctypes.byref(S), 4064)
    assert m >= 256 and m % 256 == 0
    assert lib.kv_page_append_ws() == 256 and lib.kv_topk_select_ws() == 256


def test_allocator_free_list_and_refcounts(lib):
    a = kvq.Allocator(10, seed=0)
    assert a.alloc(3) == [0, 1, 2]
    assert a.num_free() == 7
    a.ref(1)
    assert a.refcount(1) == 2
    a.free(1)
    assert a.refcount(1) == 1 and a.num_free() == 7
    a.free(1)
    assert a.refcount(1) == 0 and a.num_free() == 8
    assert a.alloc(1) == [1]          # most recently freed page is reused first
    with pytest.raises(kvq.KvqError) as e:
        a.alloc(8)
    assert e.value.code == _abi.KVQ_ERR_NO_SPACE
    assert a.num_free() == 7          # a failed allocation takes nothing
    with pytest.raises(kvq.KvqError):
        a.free(9)                     # never allocated
    with pytest.raises(kvq.KvqError):
        a.ref(9)


def test_allocator_shuffled_is_a_permutation(lib):
    a = kvq.Allocator(1000, seed=42)
    ids = a.alloc(1000)
    assert sorted(ids) == list(range(1000)) and ids != list(range(1000))
    b = kvq.Allocator(1000, seed=42)
    assert b.alloc(1000) == ids        # seeded: reproducible


@pytest.mark.parametrize("bits", [1, 2, 4, 8])
def test_code_layout_is_a_packing(bits):
    """Every (token, channel) code of a K row and a V page block owns its own
    bits, inside the block, with the two codes of a pair in the two half words."""
    from kvq_format import k_code_pos, v_code_pos
    seen = set()
    for c in range(128):
        w, b = k_code_pos(c, bits)
        assert 0 <= w < 4 * bits and 0 <= b and b % 16 + bits <= 16
        seen.update((w, b + i) for i in range(bits))
        if c % 2 == 0:
            assert k_code_pos(c + 1, bits) == (w, b + 16)
    assert len(seen) == 128 * bits
    seen = set()
    for tok in range(16):
        for d in range(128):
            w, b = v_code_pos(tok, d, bits)
            assert 0 <= w < 64 * bits and b % 16 + bits <= 16
            seen.update((w, b + i) for i in range(bits))
            if tok % 2 == 0:
                assert v_code_pos(tok + 1, d, bits) == (w, b + 16)
    assert len(seen) == 16 * 128 * bits


def test_classify_heads_matches_the_oracle(lib):
    """Head-level classification (TailorKV section 6) is host code: it equals the oracle's rule."""
    import numpy as np

    from oracle import kvq_oracle as O
    rng = np.random.default_rng(4)
    for Hq, Hkv in ((8, 2), (32, 8), (4, 4), (8, 1)):
        for _ in range(20):
            P = (rng.random(Hq) * 32).astype(np.float32)
            got = kvq.kvq_classify_heads(P.tolist(), Hq, Hkv, 32, 0.2)
            assert got == [int(x) for x in O.classify_heads(P.astype(np.float64), 32, 0.2, Hkv)]
    assert kvq.kvq_classify_heads([8.0, 8.0], 2, 1, 32, 0.25) == [0]      # equal: not above
    assert lib.kvq_classify_heads(None, 2, 1, 32, 0.2, None) == _abi.KVQ_ERR_INVALID_ARG


def test_outlier_and_dense_pref_validation(lib):
    """The outlier-isolation entries, the mixed layer's and the dense-preference workspace sizes:
    bad arguments rejected on the host before any launch."""
    by = ctypes.byref
    L4 = kvq.make_layout(8, 2, 4, 32)
    L2 = kvq.make_layout(8, 2, 2, 64)
    S = _abi.Seqs(None, None, 0, 8, 100, 0)
    fake = 1 << 20            # a 16-byte aligned non-NULL address: never dereferenced by these checks
    ws = lib.kv_outlier_channels_ws(by(L4))
    assert ws == 256 + 2 * 4 * 128 * 8
    H, d = 2, 128
    for n_out in (0, 9):
        assert lib.kv_outlier_channels(by(L4), fake, 10, H * d, n_out, fake, None, fake, ws, None) \
            == _abi.KVQ_ERR_INVALID_ARG
    assert lib.kv_outlier_channels(by(L4), fake, (1 << 22) + 1, H * d, 1, fake, None, fake, ws, None) \
        == _abi.KVQ_ERR_INVALID_ARG
    assert lib.kv_outlier_channels(by(L4), fake, 10, H * d - 8, 1, fake, None, fake, ws, None) \
        == _abi.KVQ_ERR_INVALID_ARG
    assert lib.kv_outlier_channels(by(L4), fake + 8, 10, H * d, 1, fake, None, fake, ws, None) \
        == _abi.KVQ_ERR_INVALID_ARG                                   # k not 16-byte aligned
    assert lib.kv_outlier_channels(by(L4), fake, 10, H * d, 1, fake, None, fake, ws - 8, None) \
        == _abi.KVQ_ERR_INVALID_ARG                                   # workspace too small
    P = _abi.Pool(8, 1, 0, fake, fake, fake, fake, fake, None, None, None, None)
    # isolation and the outlier attention: 4- and 8-bit layers only, 1 <= n_out <= 8
    assert lib.kv_outlier_isolate(by(L2), by(P), by(S), 0, 0, 64, fake, H * d, 1, fake, fake, None) \
        == _abi.KVQ_ERR_UNSUPPORTED
    assert lib.kv_outlier_isolate(by(L4), by(P), by(S), 0, 0, 64, fake, H * d, 9, fake, fake, None) \
        == _abi.KVQ_ERR_INVALID_ARG
    S0 = _abi.Seqs(None, None, 0, 0, 0, 0)
    wa = lib.kv_decode_attn_quant_ws(by(L4), by(S0))
    assert lib.kv_decode_attn_quant_outlier(by(L2), by(P), by(S0), fake, 1, fake, fake, fake, fake, wa, None) \
        == _abi.KVQ_ERR_UNSUPPORTED
    assert lib.kv_decode_attn_quant_outlier(by(L4), by(P), by(S0), fake, 9, fake, fake, fake, fake, wa, None) \
        == _abi.KVQ_ERR_INVALID_ARG
    assert lib.kv_decode_attn_quant_outlier(by(L4), by(P), by(S0), fake, 1, fake, None, fake, fake, wa, None) \
        == _abi.KVQ_ERR_INVALID_ARG                                   # NULL k_out
    assert lib.kv_decode_attn_quant_outlier(by(L4), by(P), by(S0), fake, 1, fake, fake + 8, fake, fake, wa, None) \
        == _abi.KVQ_ERR_INVALID_ARG                                   # k_out not 16-byte aligned
    # the mixed layer's workspace holds the dense kv heads' split records; the dense-preference
    # workspace holds the score matrix (batch x H_q x n_q x max_len rounded up to 128, fp32)
    L16 = kvq.make_layout(32, 8, 16)
    S1 = _abi.Seqs(None, None, 1, 8200, 131136, 0)
    m = lib.kv_mixed_layer_decode_ws(by(L16), by(S1))
    assert m % 256 == 0 and m > 8 * 128 * 4 * (4 + 128) * 4
    n = lib.kv_dense_pref_score_ws(by(L16), by(S1), 32)
    assert n % 256 == 0 and n >= 32 * 32 * 131200 * 4
    # (q heads per kv head) x n_q above 512 rows: not supported
    Lw = kvq.make_layout(32, 2, 16)
    S2 = _abi.Seqs(None, None, 1, 64, 1024, 0)
    Pk = _abi.Pool(64, 1, 1024, None, None, None, None, None, fake, fake, None, None)
    nw = lib.kv_dense_pref_score_ws(by(Lw), by(S2), 64)
    assert lib.kv_dense_pref_score(by(Lw), by(Pk), by(S2), fake, 64, 8, fake, fake, nw, None) \
        == _abi.KVQ_ERR_UNSUPPORTED


def _plan(lib, L, S, noalloc=0):
    n, g = ctypes.c_int32(), ctypes.c_int32()
    st = lib.kv_decode_attn_quant_plan(ctypes.byref(L), ctypes.byref(S), noalloc, ctypes.byref(n), ctypes.byref(g))
    assert st == _abi.KVQ_OK, _abi.last_error()
    return n.value, g.value


def test_quant_attention_split_plans(lib):
    """The context split of the quantized attention (a host-only query) covers every 64-token
    group exactly once, (n - 1) cps < groups <= n cps, in its three regimes: one long sequence
    (splits fill one wave of resident CTAs: the 1-bit 128K layer takes more than 16 groups a
    split, so each of a CTA's 16 warps loops through its double buffer), a batch of many units
    (a fixed 32 groups a split) and a short sequence (one split); the allocation-free plan never
    takes more splits than the workspace plan."""
    cases = [  # (layout, batch, longest sequence)
        (kvq.make_layout(32, 8, 1, 64), 1, 131072 + 37),
        (kvq.make_layout(32, 32, 4, 32), 16, 32768),
        (kvq.make_layout(8, 2, 1, 64), 1, 100),
    ]
    plans = []
    for L, B, T in cases:
        S = _abi.Seqs(None, None, B, (T + 15) // 16, T, 0)
        groups = (T + 63) // 64
        n, cps = _plan(lib, L, S)
        assert n >= 1 and cps >= 1 and (n - 1) * cps < groups <= n * cps, (n, cps, groups)
        n2, cps2 = _plan(lib, L, S, 1)
        assert 1 <= n2 <= n and (n2 - 1) * cps2 < groups <= n2 * cps2, (n2, cps2, groups)
        plans.append((n, cps))
    assert plans[0][1] > 16
    assert plans[1][1] == 32
    assert plans[2] == (1, 2)
