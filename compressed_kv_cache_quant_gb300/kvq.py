"""Python binding of libkvq with the C ABI's names (include/kvq.h).

Marshalling only: tensors become device pointers, structs are passed by
reference, a non-zero status raises KvqError.  Device memory comes from
PyTorch (caller-owned); the library never allocates.

Helpers:
  LayerCache -- allocates one layer's pool arrays as torch tensors and holds
                the kvq_layout / kvq_pool descriptors;
  Batch      -- block table + sequence lengths (kvq_seqs);
  Workspace  -- a zero-filled, 256-byte aligned device buffer;
  Allocator  -- the host page allocator (free list + reference counts).
"""
from __future__ import annotations

import ctypes

import torch

from . import _abi
from ._abi import (BITS_E4M3, BLOCK_TOKENS, HEAD_DIM, K_GROUP_TOKENS, V_SYMMETRIC, KvqError, Layout, Pool,  # noqa: F401
                   Seqs, check, lib)


def _p(x):
    """Device/host pointer of a tensor (None stays NULL; ints pass through)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _s(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ref(x):
    return ctypes.byref(x.c if hasattr(x, "c") else x)


# ------------------------------------------------------------------ descriptors

def make_layout(n_q_heads, n_kv_heads, bits, v_group_dims=64):
    return Layout(HEAD_DIM, n_q_heads, n_kv_heads, BLOCK_TOKENS, bits, K_GROUP_TOKENS, v_group_dims)


class LayerCache:
    """Device storage of one layer (torch tensors) plus its kvq_layout/kvq_pool."""

    def __init__(self, n_q_heads, n_kv_heads, bits, num_blocks, max_seqs, v_group_dims=64, t_cap=0,
                 device="cuda"):
        self.layout = make_layout(n_q_heads, n_kv_heads, bits, v_group_dims)
        H, d, P = n_kv_heads, HEAD_DIM, BLOCK_TOKENS
        self.bits, self.H, self.num_blocks, self.max_seqs, self.t_cap = bits, H, num_blocks, max_seqs, t_cap
        z = lambda shape, dt: torch.zeros(shape, dtype=dt, device=device)  # noqa: E731
        self.k_codes = self.v_codes = self.k_sz = self.v_sz = self.k_tail = None
        self.k16 = self.v16 = self.kT = self.k_absmax = None
        if bits == _abi.BITS_E4M3:
            self.k_codes = z((num_blocks, H, P, d), torch.uint8)
            self.v_codes = z((num_blocks, H, P, d), torch.uint8)
        elif bits == 16:
            self.k16 = z((num_blocks, H, P, d), torch.float16)
            self.v16 = z((num_blocks, H, P, d), torch.float16)
            if t_cap:
                self.kT = z((max_seqs, H, d, t_cap), torch.float16)
                self.k_absmax = z((max_seqs, H, d), torch.float32)
        else:
            R = d * (bits & 0xFF) // 8
            self.k_codes = z((num_blocks, H, P, R), torch.uint8)
            self.v_codes = z((num_blocks, H, P, R), torch.uint8)
            self.k_sz = z((num_blocks, H, d, 2), torch.float16)
            self.v_sz = z((num_blocks, H, P, d // v_group_dims, 2), torch.float16)
            self.k_tail = z((max_seqs, H, K_GROUP_TOKENS, d), torch.float16)
        self.c = Pool(num_blocks, max_seqs, t_cap, _p(self.k_codes), _p(self.v_codes), _p(self.k_sz),
                      _p(self.v_sz), _p(self.k_tail), _p(self.k16), _p(self.v16), _p(self.kT),
                      _p(self.k_absmax))


class Batch:
    """Block table + sequence lengths of a batch (kvq_seqs)."""

    def __init__(self, block_table, seq_lens, max_len):
        assert block_table.dtype == torch.int32 and seq_lens.dtype == torch.int32
        self.block_table = block_table.contiguous()
        self.seq_lens = seq_lens.contiguous()
        self.max_len = int(max_len)
        B, mb = self.block_table.shape
        self.c = Seqs(_p(self.block_table), _p(self.seq_lens), B, mb, self.max_len, 0)

    @property
    def batch(self):
        return self.c.batch


class Workspace:
    """Zero-filled device workspace of `nbytes` (rounded to 256)."""

    def __init__(self, nbytes, device="cuda"):
        n = max(256, (int(nbytes) + 255) // 256 * 256)
        self.t = torch.zeros(n + 256, dtype=torch.uint8, device=device)
        off = (-self.t.data_ptr()) % 256
        self.ptr = self.t.data_ptr() + off
        self.nbytes = n


class Allocator:
    """Host page allocator (free list, reference counts for shared pages)."""

    def __init__(self, num_blocks, seed=0):
        self.h = lib().kvq_alloc_create(int(num_blocks), int(seed))
        if not self.h:
            raise KvqError(_abi.KVQ_ERR_INVALID_ARG, "kvq_alloc_create", _abi.last_error())

    def alloc(self, n):
        ids = (ctypes.c_int32 * max(n, 1))()
        check(lib().kvq_block_alloc(self.h, int(n), ids), "kvq_block_alloc")
        return [ids[i] for i in range(n)]

    def ref(self, page):
        check(lib().kvq_block_ref(self.h, int(page)), "kvq_block_ref")

    def free(self, page):
        check(lib().kvq_block_free(self.h, int(page)), "kvq_block_free")

    def refcount(self, page):
        r = lib().kvq_block_refcount(self.h, int(page))
        if r < 0:
            raise KvqError(r, "kvq_block_refcount", _abi.last_error())
        return r

    def num_free(self):
        return lib().kvq_alloc_num_free(self.h)

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            lib().kvq_alloc_destroy(h)
            self.h = None


# ------------------------------------------------------------------ the C ABI, same names

def kv_quant_pack(cache, seqs, seq, t_start, n_tokens, k, v, stride_t=None, stream=None):
    if stride_t is None:
        stride_t = cache.H * HEAD_DIM
    return check(lib().kv_quant_pack(_ref(cache.layout), _ref(cache), _ref(seqs), int(seq), int(t_start),
                                      int(n_tokens), _p(k), _p(v), int(stride_t), _s(stream)), "kv_quant_pack")


def kv_page_append_ws():
    return lib().kv_page_append_ws()


def kv_page_append(cache, seqs, k_new, v_new, ws, stream=None):
    return check(lib().kv_page_append(_ref(cache.layout), _ref(cache), _ref(seqs), _p(k_new), _p(v_new), ws.ptr,
                                      ws.nbytes, _s(stream)), "kv_page_append")


def kv_decode_attn_quant_ws(cache, seqs):
    return lib().kv_decode_attn_quant_ws(_ref(cache.layout), _ref(seqs))


def kv_decode_attn_quant(cache, seqs, q, out, ws, stream=None):
    return check(lib().kv_decode_attn_quant(_ref(cache.layout), _ref(cache), _ref(seqs), _p(q), _p(out), ws.ptr,
                                            ws.nbytes, _s(stream)), "kv_decode_attn_quant")


def kv_decode_attn_quant_noalloc(cache, seqs, q, out, stream=None):
    """kv_decode_attn_quant with the library's built-in scratch array instead of a
    workspace, for callers that may not allocate device memory."""
    return check(lib().kv_decode_attn_quant_noalloc(_ref(cache.layout), _ref(cache), _ref(seqs), _p(q), _p(out),
                                                    _s(stream)), "kv_decode_attn_quant_noalloc")


def kv_decode_attn_quant_noalloc_max_scratch():
    return lib().kv_decode_attn_quant_noalloc_max_scratch()


def kv_decode_attn_quant_plan(cache, seqs, noalloc=False):
    """(n_splits, groups_per_split) the quantized attention uses for this batch."""
    n, g = ctypes.c_int32(0), ctypes.c_int32(0)
    check(lib().kv_decode_attn_quant_plan(_ref(cache.layout), _ref(seqs), int(bool(noalloc)), ctypes.byref(n),
                                          ctypes.byref(g)), "kv_decode_attn_quant_plan")
    return n.value, g.value


def _layout_of(x):
    return x.layout if hasattr(x, "layout") else x


def kv_outlier_channels_ws(layout):
    """Workspace bytes of kv_outlier_channels (`layout`: a Layout or a cache)."""
    return lib().kv_outlier_channels_ws(ctypes.byref(_layout_of(layout)))


def kv_outlier_channels(layout, k, n_tokens, n_out, out_ch, ws, var=None, stride_t=None, stream=None):
    """The n_out largest-variance key channels per kv head of k [n_tokens][H_kv][d] (fp16)
    into out_ch [H_kv][n_out] (int32), optionally the variances into var [H_kv][d] (fp64)."""
    st = stride_t if stride_t is not None else k.stride(0)
    return check(lib().kv_outlier_channels(ctypes.byref(_layout_of(layout)), _p(k), n_tokens, st, n_out, _p(out_ch),
                                           _p(var), ws.ptr, ws.nbytes, _s(stream)), "kv_outlier_channels")


def kv_outlier_isolate(cache, seqs, seq, t_start, n_tokens, k, n_out, out_ch, k_out, stride_t=None, stream=None):
    st = stride_t if stride_t is not None else k.stride(0)
    return check(lib().kv_outlier_isolate(_ref(cache.layout), _ref(cache), _ref(seqs), seq, t_start, n_tokens, _p(k),
                                          st, n_out, _p(out_ch), _p(k_out), _s(stream)), "kv_outlier_isolate")


def kv_outlier_append_ws():
    return lib().kv_outlier_append_ws()


def kv_outlier_append(cache, seqs, n_out, out_ch, k_out, ws, stream=None):
    return check(lib().kv_outlier_append(_ref(cache.layout), _ref(cache), _ref(seqs), n_out, _p(out_ch), _p(k_out),
                                         ws.ptr, ws.nbytes, _s(stream)), "kv_outlier_append")


def kv_decode_attn_quant_outlier(cache, seqs, q, n_out, out_ch, k_out, out, ws, stream=None):
    return check(lib().kv_decode_attn_quant_outlier(_ref(cache.layout), _ref(cache), _ref(seqs), _p(q), n_out,
                                                    _p(out_ch), _p(k_out), _p(out), ws.ptr, ws.nbytes, _s(stream)),
                 "kv_decode_attn_quant_outlier")


def kv_critical_score(cache, seqs, q, n_crit, crit, scores, score_stride=None, stream=None):
    if score_stride is None:
        score_stride = scores.shape[-1]
    return check(lib().kv_critical_score(_ref(cache.layout), _ref(cache), _ref(seqs), _p(q), int(n_crit), _p(crit),
                                         _p(scores), int(score_stride), _s(stream)), "kv_critical_score")


def kv_group_critical_score(cache, seqs, q, n_crit, crit, scores, score_stride=None, stream=None):
    if score_stride is None:
        score_stride = scores.shape[-1]
    return check(lib().kv_group_critical_score(_ref(cache.layout), _ref(cache), _ref(seqs), _p(q), int(n_crit),
                                               _p(crit), _p(scores), int(score_stride), _s(stream)),
                 "kv_group_critical_score")


def kv_append_critical_score_ws():
    return lib().kv_append_critical_score_ws()


def kv_append_critical_score(cache, seqs, k_new, v_new, q, n_crit, crit, scores, hist, n_sink, window, ws,
                             score_stride=None, stream=None):
    if score_stride is None:
        score_stride = scores.shape[-1]
    return check(lib().kv_append_critical_score(_ref(cache.layout), _ref(cache), _ref(seqs), _p(k_new), _p(v_new),
                                                _p(q), int(n_crit), _p(crit), _p(scores), int(score_stride),
                                                _p(hist), int(n_sink), int(window), ws.ptr, ws.nbytes, _s(stream)),
                 "kv_append_critical_score")


def kv_select_sparse_attn_ws():
    return lib().kv_select_sparse_attn_ws()


def kv_select_sparse_attn(cache, seqs, q, scores, hist, k_fixed, ratio, n_sink, window, sel, sel_count, out, ws,
                          score_stride=None, stream=None):
    if score_stride is None:
        score_stride = scores.shape[-1]
    sel_cap = int(sel.shape[-1]) if sel is not None else 0
    return check(lib().kv_select_sparse_attn(_ref(cache.layout), _ref(cache), _ref(seqs), _p(q), _p(scores),
                                             int(score_stride), _p(hist), int(k_fixed), float(ratio), int(n_sink),
                                             int(window), _p(sel), sel_cap, _p(sel_count), _p(out), ws.ptr,
                                             ws.nbytes, _s(stream)), "kv_select_sparse_attn")


def kv_sparse_layer_decode_ws():
    return lib().kv_sparse_layer_decode_ws()


def kv_sparse_layer_decode(cache, seqs, k_new, v_new, q, n_crit, k_fixed, ratio, n_sink, window, out, ws,
                           scores=None, sel=None, sel_count=None, stream=None):
    stride = int(scores.shape[-1]) if scores is not None else 0
    sel_cap = int(sel.shape[-1]) if sel is not None else 0
    return check(lib().kv_sparse_layer_decode(_ref(cache.layout), _ref(cache), _ref(seqs), _p(k_new), _p(v_new),
                                              _p(q), int(n_crit), int(k_fixed), float(ratio), int(n_sink),
                                              int(window), _p(scores), stride, _p(sel), sel_cap, _p(sel_count),
                                              _p(out), ws.ptr, ws.nbytes, _s(stream)), "kv_sparse_layer_decode")


def kv_mixed_layer_decode_ws(cache, seqs):
    return lib().kv_mixed_layer_decode_ws(_ref(cache.layout), _ref(seqs))


def kv_mixed_layer_decode(cache, seqs, k_new, v_new, q, n_crit, k_fixed, ratio, n_sink, window, dense, out, ws,
                          sel=None, sel_count=None, stream=None):
    sel_cap = int(sel.shape[-1]) if sel is not None else 0
    return check(lib().kv_mixed_layer_decode(_ref(cache.layout), _ref(cache), _ref(seqs), _p(k_new), _p(v_new),
                                             _p(q), int(n_crit), int(k_fixed), float(ratio), int(n_sink), int(window),
                                             _p(dense), _p(sel), sel_cap, _p(sel_count), _p(out), ws.ptr, ws.nbytes,
                                             _s(stream)), "kv_mixed_layer_decode")


def kvq_classify_heads(P, n_q_heads, n_kv_heads, n_q, tau):
    """Per kv head: 1 if its q heads' mean dense-preference score over n_q exceeds tau."""
    Pa = (ctypes.c_float * n_q_heads)(*[float(x) for x in P])
    out = (ctypes.c_int32 * n_kv_heads)()
    r = lib().kvq_classify_heads(Pa, int(n_q_heads), int(n_kv_heads), int(n_q), float(tau), out)
    if r < 0:
        raise KvqError(r, "kvq_classify_heads", _abi.last_error())
    return [int(out[i]) for i in range(n_kv_heads)]


def kv_topk_select_ws():
    return lib().kv_topk_select_ws()


def kv_topk_select(seqs, n_heads, scores, k_fixed, ratio, n_sink, window, sel, sel_count, ws, score_stride=None,
                   stream=None):
    if score_stride is None:
        score_stride = scores.shape[-1]
    return check(lib().kv_topk_select(_ref(seqs), int(n_heads), _p(scores), int(score_stride), int(k_fixed),
                                      float(ratio), int(n_sink), int(window), _p(sel), int(sel.shape[-1]),
                                      _p(sel_count), ws.ptr, ws.nbytes, _s(stream)), "kv_topk_select")


def kv_block_select_ws(seqs, n_heads, block_tokens):
    return lib().kv_block_select_ws(_ref(seqs), int(n_heads), int(block_tokens))


def kv_block_select(seqs, n_heads, scores, n_keep_fixed, ratio, n_sink, window, block_tokens, sel, sel_count, ws,
                    score_stride=None, stream=None):
    if score_stride is None:
        score_stride = scores.shape[-1]
    return check(lib().kv_block_select(_ref(seqs), int(n_heads), _p(scores), int(score_stride), int(n_keep_fixed),
                                       float(ratio), int(n_sink), int(window), int(block_tokens), _p(sel),
                                       int(sel.shape[-1]), _p(sel_count), ws.ptr, ws.nbytes, _s(stream)),
                 "kv_block_select")


def kv_sparse_attn_ws(cache, seqs, sel_cap):
    return lib().kv_sparse_attn_ws(_ref(cache.layout), _ref(seqs), int(sel_cap))


def kv_sparse_attn(cache, seqs, q, sel, sel_count, sel_per_kv_head, out, probs, ws, stream=None):
    return check(lib().kv_sparse_attn(_ref(cache.layout), _ref(cache), _ref(seqs), _p(q), _p(sel),
                                      int(sel.shape[-1]), _p(sel_count), int(sel_per_kv_head), _p(out), _p(probs),
                                      ws.ptr, ws.nbytes, _s(stream)), "kv_sparse_attn")


def kv_h2o_accumulate_ws():
    return lib().kv_h2o_accumulate_ws()


def kv_h2o_accumulate(cache, seqs, probs, retained, retained_count, cum, budget, n_sink, window, new_pos, n_evicted,
                      ws, stream=None):
    return check(lib().kv_h2o_accumulate(_ref(cache.layout), _ref(seqs), _p(probs), _p(retained),
                                         _p(retained_count), _p(cum), int(retained.shape[-1]), int(budget),
                                         int(n_sink), int(window), _p(new_pos), _p(n_evicted), ws.ptr, ws.nbytes,
                                         _s(stream)), "kv_h2o_accumulate")


def kv_dense_pref_score_ws(cache, seqs, n_q):
    return lib().kv_dense_pref_score_ws(_ref(cache.layout), _ref(seqs), int(n_q))


def kv_dense_pref_score(cache, seqs, q_recent, n_q, topk, P, ws, stream=None):
    return check(lib().kv_dense_pref_score(_ref(cache.layout), _ref(cache), _ref(seqs), _p(q_recent), int(n_q),
                                           int(topk), _p(P), ws.ptr, ws.nbytes, _s(stream)), "kv_dense_pref_score")


def kv_offload_gather_ws():
    return lib().kv_offload_gather_ws()


def kv_offload_gather(src_k, src_v, src_stride_h, src_rows, n_heads, sel, sel_count, dst_k, dst_v, ws, stream=None):
    return check(lib().kv_offload_gather(_p(src_k), _p(src_v), int(src_stride_h), int(src_rows), int(n_heads),
                                         _p(sel), int(sel.shape[-1]), _p(sel_count), _p(dst_k), _p(dst_v), ws.ptr,
                                         ws.nbytes, _s(stream)), "kv_offload_gather")


def kvq_seq_lens_add(seq_lens, delta, stream=None):
    return check(lib().kvq_seq_lens_add(_p(seq_lens), int(seq_lens.numel()), int(delta), _s(stream)),
                 "kvq_seq_lens_add")


def kv_page_copy(cache, src, dst, stream=None):
    return check(lib().kv_page_copy(_ref(cache.layout), _ref(cache), int(src), int(dst), _s(stream)),
                 "kv_page_copy")


def kvq_check(ws, stream=None):
    return check(lib().kvq_check(ws.ptr, _s(stream)), "kvq_check")


def kvq_selftest_bounded_wait(ws, stream=None):
    """Runs the library's bounded mbarrier wait on a barrier nothing completes (see kvq.h)."""
    return check(lib().kvq_selftest_bounded_wait(ws.ptr, ws.nbytes, _s(stream)), "kvq_selftest_bounded_wait")


def kvq_read_path_counters(ws, stream=None):
    """The workspace's diagnostic path counters (KVQ_PATH_*), read and cleared."""
    out = (ctypes.c_uint32 * _abi.N_PATH_COUNTERS)()
    check(lib().kvq_read_path_counters(ws.ptr, out, _s(stream)), "kvq_read_path_counters")
    return [int(out[i]) for i in range(_abi.N_PATH_COUNTERS)]
