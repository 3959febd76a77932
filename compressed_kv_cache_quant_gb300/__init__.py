"""GB300-native compressed-KV decode attention (libkvq) and its Python binding.

The hot path runs in hand-written CUDA kernels for sm_103a inside libkvq.so
(built in-tree by ``compressed_kv_cache_quant_gb300.build``); this package
only marshals arguments to the C ABI declared in include/kvq.h.
"""
from . import _abi  # noqa: F401
from .kvq import (Allocator, Batch, KvqError, LayerCache, Workspace, kv_append_critical_score,  # noqa: F401
                  kv_append_critical_score_ws, kv_block_select, kv_block_select_ws, kv_critical_score, kv_select_sparse_attn, kv_select_sparse_attn_ws,
                  kv_decode_attn_quant, kv_decode_attn_quant_ws, kv_dense_pref_score, kv_dense_pref_score_ws,
                  kv_h2o_accumulate, kv_h2o_accumulate_ws, kv_offload_gather, kv_offload_gather_ws, kv_page_append,
                  kv_page_append_ws, kv_page_copy, kv_quant_pack, kv_sparse_attn, kv_sparse_attn_ws, kv_sparse_layer_decode,
                  kv_sparse_layer_decode_ws, kv_topk_select,
                  kv_topk_select_ws, kvq_check, kvq_seq_lens_add, make_layout)
