"""GB300-native DeepSeek-sparse-attention indexer candidate selection.

The work runs in hand-written sm_103a CUDA kernels behind a C ABI
(include/dsa_select.h, built by ``build.build()``); this package is the thin
Python binding over it.
"""
from .binding import (attention_cfg, dsa_attention_cfg, dsa_group_union, dsa_sparse_attention,
                      dsa_group_union_ranges, dsa_sparse_attention_ranges,
                      dsa_sparse_attention_ranges_workspace, ranges_attention_cfg,
                      dsa_sparse_attention_status, dsa_sparse_attention_workspace, DSA_ERR_CUDA, DSA_ERR_INVALID_ARG, DSA_ERR_TIMEOUT, DSA_ERR_UNSUPPORTED,
                      DSA_OK, NOALLOC_SCRATCH_BYTES, DsaSelectError, EXPORTS, Plan,
                      dsa_candidate_select,
                      dsa_combine_window, dsa_indexer_cfg, dsa_indexer_logits,
                      dsa_indexer_select, dsa_indexer_select_noalloc,
                      dsa_indexer_select_workspace, dsa_indexer_status,
                      dsa_plan_desc, dsa_row_topk, dsa_select_cfg, dsa_select_init,
                      dsa_select_topk, load, make_cfg, status_string)
from .build import LIB_PATH, build
from .sharded import Shard, ShardedSelector, shard_rows

__all__ = ["DSA_OK", "DSA_ERR_INVALID_ARG", "DSA_ERR_UNSUPPORTED", "DSA_ERR_CUDA",
           "DSA_ERR_TIMEOUT", "DsaSelectError", "EXPORTS", "Plan", "dsa_select_cfg",
           "dsa_plan_desc", "make_cfg", "dsa_select_init", "dsa_candidate_select",
           "dsa_row_topk", "dsa_select_topk", "dsa_combine_window", "dsa_indexer_cfg",
           "dsa_indexer_logits", "dsa_indexer_select", "dsa_indexer_select_workspace",
           "dsa_indexer_select_noalloc", "NOALLOC_SCRATCH_BYTES",
           "dsa_indexer_status", "status_string", "load", "build", "LIB_PATH",
           "Shard", "ShardedSelector", "shard_rows", "attention_cfg", "dsa_attention_cfg",
           "dsa_group_union", "dsa_sparse_attention_workspace", "dsa_sparse_attention",
           "dsa_sparse_attention_status", "ranges_attention_cfg", "dsa_sparse_attention_ranges_workspace",
           "dsa_group_union_ranges", "dsa_sparse_attention_ranges"]
