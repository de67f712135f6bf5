"""Chunked-prefill attention over a paged KV cache for NVIDIA GB300 (sm_103a).

The compute lives in libcpsa.so (hand-written CUDA, C ABI in include/cpsa.h);
this package is its Python binding plus host-side orchestration:

  cpp_kv_cache_write        slot_mapping scatter of the new tokens' K/V
  cpp_chunked_prefill_attn  causal attention of prefill chunks and decode rows
  cpp_chunked_prefill_attn_write_kv
                            the KV write fused into that attention call
  cpp_split_microbatch      balanced micro-batch split point
  cpp_plan_chunk_sizes      dynamic chunk planner (quadratic latency model)
  OnlineChunker             online chunk-size controller (windowed refit of f(C, H))
  BatchScheduler            token-budget batch builder with page allocation
  AttentionStep             one step (KV write + attention) with its workspace,
                            on one stream or as two micro-batches on two streams
"""
from ._lib import (  # noqa: F401
    CpsaError, load, cpp_kv_cache_write, cpp_attn_workspace_bytes, cpp_attn_workspace_min_bytes,
    cpp_chunked_prefill_attn, cpp_chunked_prefill_attn_events, cpp_chunked_prefill_attn_noalloc,
    cpp_noalloc_scratch_address,
    cpp_chunked_prefill_attn_write_kv,
    cpp_split_microbatch, cpp_read_device_error, cpp_get_device_error, cpp_plan_chunk_sizes,
    cpp_fit_latency_quadratic, cpp_fit_latency_two_var, cpp_selftest_exp2, cpp_selftest_wait_timeout,
    OnlineChunker, BatchScheduler,
    DEV_SLOT_OUT_OF_RANGE, DEV_PAGE_OUT_OF_RANGE, DEV_SEQ_LT_QUERY, DEV_TOKENS_MISMATCH, DEV_SEQ_GT_TABLE,
    DEV_SPLITS_CLAMPED, DEV_WAIT_TIMEOUT,
)
from .step import AttentionStep  # noqa: F401
