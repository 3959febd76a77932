"""ctypes view of the libkvq C ABI (include/kvq.h): structs, prototypes, loader.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Importing this module does not load the library; ``lib()`` does, and
raises if libkvq.so has not been built -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_double, c_int, c_int32, c_int64, c_size_t, c_uint32, c_uint64, c_void_p

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvq.so")

KVQ_OK = 0
KVQ_ERR_INVALID_ARG = -1
KVQ_ERR_UNSUPPORTED = -2
KVQ_ERR_CUDA = -3
KVQ_ERR_NO_SPACE = -4
KVQ_ERR_TIMEOUT = -5
KVQ_ERR_DEVICE_CHECK = -6
ABI_VERSION = 1

HEAD_DIM = 128
BLOCK_TOKENS = 16
BITS_E4M3 = 0xE4          # kvq_layout.bits of an FP8 E4M3 layer
V_SYMMETRIC = 0x100       # or-ed into kvq_layout.bits: V quantized symmetrically
K_GROUP_TOKENS = 64

N_PATH_COUNTERS = 4
PATH_LISTED, PATH_COMPACTED, PATH_RADIX_PASSES = 0, 1, 2


class KvqError(RuntimeError):
    def __init__(self, code, fn, msg):
        super().__init__(f"{fn} failed with status {code}: {msg}")
        self.code = code
        self.fn = fn


class Layout(ctypes.Structure):
    _fields_ = [("head_dim", c_int32), ("n_q_heads", c_int32), ("n_kv_heads", c_int32),
                ("block_tokens", c_int32), ("bits", c_int32), ("k_group_tokens", c_int32),
                ("v_group_dims", c_int32)]


class Pool(ctypes.Structure):
    _fields_ = [("num_blocks", c_int64), ("max_seqs", c_int32), ("t_cap", c_int32),
                ("k_codes", c_void_p), ("v_codes", c_void_p), ("k_sz", c_void_p), ("v_sz", c_void_p),
                ("k_tail", c_void_p), ("k16", c_void_p), ("v16", c_void_p), ("kT", c_void_p),
                ("k_absmax", c_void_p)]


class Seqs(ctypes.Structure):
    _fields_ = [("block_table", c_void_p), ("seq_lens", c_void_p), ("batch", c_int32),
                ("max_blocks", c_int32), ("max_len", c_int32), ("reserved", c_int32)]


PL, PP, PS = POINTER(Layout), POINTER(Pool), POINTER(Seqs)
VP = c_void_p

# name -> (restype, argtypes); mirrors include/kvq.h
PROTOTYPES = {
    "kvq_last_error": (c_char_p, []),
    "kvq_version": (c_int, []),
    "kv_quant_pack": (c_int, [PL, PP, PS, c_int32, c_int64, c_int64, VP, VP, c_int64, VP]),
    "kv_page_append": (c_int, [PL, PP, PS, VP, VP, VP, c_size_t, VP]),
    "kv_page_append_ws": (c_size_t, []),
    "kv_decode_attn_quant": (c_int, [PL, PP, PS, VP, VP, VP, c_size_t, VP]),
    "kv_decode_attn_quant_ws": (c_size_t, [PL, PS]),
    "kv_decode_attn_quant_noalloc": (c_int, [PL, PP, PS, VP, VP, VP]),
    "kv_decode_attn_quant_noalloc_max_scratch": (c_size_t, []),
    "kv_decode_attn_quant_plan": (c_int, [PL, PS, c_int32, POINTER(c_int32), POINTER(c_int32)]),
    "kv_outlier_channels": (c_int, [PL, VP, c_int64, c_int64, c_int32, VP, VP, VP, c_size_t, VP]),
    "kv_outlier_channels_ws": (c_size_t, [PL]),
    "kv_outlier_isolate": (c_int, [PL, PP, PS, c_int32, c_int64, c_int64, VP, c_int64, c_int32, VP, VP, VP]),
    "kv_outlier_append": (c_int, [PL, PP, PS, c_int32, VP, VP, VP, c_size_t, VP]),
    "kv_outlier_append_ws": (c_size_t, []),
    "kv_decode_attn_quant_outlier": (c_int, [PL, PP, PS, VP, c_int32, VP, VP, VP, VP, c_size_t, VP]),
    "kv_critical_score": (c_int, [PL, PP, PS, VP, c_int32, VP, VP, c_int64, VP]),
    "kv_group_critical_score": (c_int, [PL, PP, PS, VP, c_int32, VP, VP, c_int64, VP]),
    "kv_topk_select": (c_int, [PS, c_int32, VP, c_int64, c_int32, c_double, c_int32, c_int32, VP, c_int32, VP,
                               VP, c_size_t, VP]),
    "kv_topk_select_ws": (c_size_t, []),
    "kv_block_select": (c_int, [PS, c_int32, VP, c_int64, c_int32, c_double, c_int32, c_int32, c_int32, VP, c_int32,
                                VP, VP, c_size_t, VP]),
    "kv_block_select_ws": (c_size_t, [PS, c_int32, c_int32]),
    "kv_append_critical_score": (c_int, [PL, PP, PS, VP, VP, VP, c_int32, VP, VP, c_int64, VP, c_int32, c_int32, VP,
                                         c_size_t, VP]),
    "kv_append_critical_score_ws": (c_size_t, []),
    "kv_select_sparse_attn": (c_int, [PL, PP, PS, VP, VP, c_int64, VP, c_int32, c_double, c_int32, c_int32, VP,
                                      c_int32, VP, VP, VP, c_size_t, VP]),
    "kv_select_sparse_attn_ws": (c_size_t, []),
    "kv_sparse_layer_decode": (c_int, [PL, PP, PS, VP, VP, VP, c_int32, c_int32, c_double, c_int32, c_int32, VP,
                                       c_int64, VP, c_int32, VP, VP, VP, c_size_t, VP]),
    "kv_sparse_layer_decode_ws": (c_size_t, []),
    "kv_mixed_layer_decode": (c_int, [PL, PP, PS, VP, VP, VP, c_int32, c_int32, c_double, c_int32, c_int32, VP, VP,
                                      c_int32, VP, VP, VP, c_size_t, VP]),
    "kv_mixed_layer_decode_ws": (c_size_t, [PL, PS]),
    "kvq_classify_heads": (c_int, [POINTER(ctypes.c_float), c_int32, c_int32, c_int32, c_double, POINTER(c_int32)]),
    "kv_sparse_attn": (c_int, [PL, PP, PS, VP, VP, c_int32, VP, c_int32, VP, VP, VP, c_size_t, VP]),
    "kv_sparse_attn_ws": (c_size_t, [PL, PS, c_int32]),
    "kv_h2o_accumulate": (c_int, [PL, PS, VP, VP, VP, VP, c_int32, c_int32, c_int32, c_int32, VP, VP, VP,
                                  c_size_t, VP]),
    "kv_h2o_accumulate_ws": (c_size_t, []),
    "kv_dense_pref_score": (c_int, [PL, PP, PS, VP, c_int32, c_int32, VP, VP, c_size_t, VP]),
    "kv_dense_pref_score_ws": (c_size_t, [PL, PS, c_int32]),
    "kv_offload_gather": (c_int, [VP, VP, c_int64, c_int64, c_int32, VP, c_int32, VP, VP, VP, VP, c_size_t, VP]),
    "kv_offload_gather_ws": (c_size_t, []),
    "kvq_seq_lens_add": (c_int, [VP, c_int32, c_int32, VP]),
    "kv_page_copy": (c_int, [PL, PP, c_int32, c_int32, VP]),
    "kvq_check": (c_int, [VP, VP]),
    "kvq_read_path_counters": (c_int, [VP, POINTER(c_uint32), VP]),
    "kvq_selftest_bounded_wait": (c_int, [VP, c_size_t, VP]),
    "kvq_alloc_create": (VP, [c_int64, c_uint64]),
    "kvq_alloc_destroy": (None, [VP]),
    "kvq_block_alloc": (c_int, [VP, c_int32, POINTER(c_int32)]),
    "kvq_block_ref": (c_int, [VP, c_int32]),
    "kvq_block_free": (c_int, [VP, c_int32]),
    "kvq_block_refcount": (c_int, [VP, c_int32]),
    "kvq_alloc_num_free": (c_int64, [VP]),
}

_lib = None


def lib():
    """The loaded libkvq (prototypes declared).  Raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with compressed_kv_cache_quant_gb300.build.build() "
                              "(or __graft_entry__.build()); there is no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in PROTOTYPES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        if L.kvq_version() != ABI_VERSION:
            raise ImportError(f"libkvq ABI version {L.kvq_version()} != {ABI_VERSION}; rebuild it")
        _lib = L
    return _lib


def last_error():
    return lib().kvq_last_error().decode(errors="replace")


def check(status, fn):
    if status != KVQ_OK:
        raise KvqError(status, fn, last_error())
    return status
