"""KV-cached grouped-query attention for GB300 (sm_103a).

The compute path lives in `libkvc.so` (hand-written CUDA kernels behind the C ABI of
`include/kvc.h`); this package only builds it and marshals arguments to it.
"""
from kv_cached_gqa_gb300._binding import (KVC_BF16, KVC_COMMITTED, KVC_F16, KVC_F32, Cache, KvcError,
                                          gqa_cached_attn, kvc_append, kvc_commit, kvc_create,
                                          kvc_layer_ptrs, kvc_nbytes, kvc_positions, kvc_seq_len,
                                          kvc_set_split_keys, kvc_status, kvc_truncate,
                                          kvc_truncate_ragged, load, synth_fill_normal)

__all__ = ["KVC_BF16", "KVC_COMMITTED", "KVC_F16", "KVC_F32", "Cache", "KvcError", "gqa_cached_attn",
           "kvc_append", "kvc_commit", "kvc_create", "kvc_layer_ptrs", "kvc_nbytes", "kvc_positions",
           "kvc_seq_len", "kvc_set_split_keys", "kvc_status", "kvc_truncate", "kvc_truncate_ragged", "load",
           "synth_fill_normal"]
