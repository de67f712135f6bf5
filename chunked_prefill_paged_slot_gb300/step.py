"""One attention step of a chunked-prefill batch: KV write, then attention
(two kernels' worth of calls, or one call with the write fused into it).

Host orchestration only (workspace ownership, streams, events, pointer
offsets); every step of the computation runs in libcpsa.so's kernels.

Two-stream mode follows the "Ascend dual-stream parallel" article, section 3.1
(split point, then token-axis tensors split at token_split and request-axis
tensors at batch_split) and 3.2 (events joining the streams): the split kernel
picks the balanced request boundary; when it allows two micro-batches, each
runs its KV write and attention on its own stream over zero-copy views, and
the caller's stream waits on both.
"""
from __future__ import annotations

import torch

from . import _lib


class AttentionStep:
    def __init__(self, num_reqs: int, num_tokens: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 max_kv_splits: int = 8, device=None, workspace_bytes: int | None = None,
                 two_stream: bool = False, balance_threshold: float = 0.1, length_threshold: int = 256,
                 fused_kv_write: bool = False):
        device = torch.device(device if device is not None else "cuda")
        self.fused_kv_write = fused_kv_write
        self.dims = (num_q_heads, num_kv_heads, head_dim)
        self.max_kv_splits = max_kv_splits
        if workspace_bytes is None:
            workspace_bytes = _lib.cpp_attn_workspace_bytes(num_reqs, num_tokens, num_q_heads, num_kv_heads,
                                                            head_dim, max_kv_splits)
        n_ws = 2 if two_stream else 1
        self.workspaces = [torch.empty(workspace_bytes, dtype=torch.uint8, device=device) for _ in range(n_ws)]
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=device)
        self.split_out = torch.zeros(3, dtype=torch.int32, device=device)
        self.split_host = torch.zeros(3, dtype=torch.int32, pin_memory=True)
        self.balance_threshold = balance_threshold
        self.length_threshold = length_threshold
        self.streams = [torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)] if two_stream else None
        self.last_split = None

    def run(self, q, k, v, slot_mapping, k_cache, v_cache, query_lens, seq_lens, block_table, out,
            scale: float = 0.0, stream=None, workspace=None):
        """KV write of the new tokens, then attention, on one stream."""
        ws = self.workspaces[0] if workspace is None else workspace
        if self.fused_kv_write:
            _lib.cpp_chunked_prefill_attn_write_kv(q, k, v, slot_mapping, k_cache, v_cache, query_lens, seq_lens,
                                                   block_table, out, ws, self.dev_err, scale=scale,
                                                   max_kv_splits=self.max_kv_splits, stream=stream)
            return
        _lib.cpp_kv_cache_write(k, v, slot_mapping, k_cache, v_cache, self.dev_err, stream=stream)
        _lib.cpp_chunked_prefill_attn(q, k_cache, v_cache, query_lens, seq_lens, block_table, out, ws,
                                      self.dev_err, scale=scale, max_kv_splits=self.max_kv_splits, stream=stream)

    def split(self, query_lens, stream=None):
        """(batch_split, token_split, use_two) from the split kernel (one small D2H read)."""
        s = stream if stream is not None else torch.cuda.current_stream()
        _lib.cpp_split_microbatch(query_lens, self.split_out, self.balance_threshold, self.length_threshold,
                                  stream=s)
        self.split_host.copy_(self.split_out, non_blocking=True)
        s.synchronize()
        b, t, use = (int(x) for x in self.split_host.tolist())
        self.last_split = (b, t, bool(use))
        return self.last_split

    def run_two_stream(self, q, k, v, slot_mapping, k_cache, v_cache, query_lens, seq_lens, block_table, out,
                       scale: float = 0.0, stream=None, split=None):
        """Split the batch and run the two micro-batches on two streams (one stream when refused).
        split: (batch_split, token_split, use_two) of this batch when already known (from split()
        on the same query_lens: it depends on the lengths alone), else computed here, which reads
        the split kernel's result back to the host."""
        if self.streams is None:
            raise _lib.CpsaError("AttentionStep was built without two_stream=True")
        main = stream if stream is not None else torch.cuda.current_stream()
        b, t, use = self.split(query_lens, stream=main) if split is None else split
        if not use:
            self.run(q, k, v, slot_mapping, k_cache, v_cache, query_lens, seq_lens, block_table, out,
                     scale=scale, stream=main)
            return False
        start = torch.cuda.Event()
        start.record(main)
        parts = [(slice(0, t), slice(0, b)), (slice(t, q.shape[0]), slice(b, query_lens.shape[0]))]
        done = []
        for (ts, rs), s, ws in zip(parts, self.streams, self.workspaces):
            s.wait_event(start)
            self.run(q[ts], k[ts], v[ts], slot_mapping[ts], k_cache, v_cache, query_lens[rs], seq_lens[rs],
                     block_table[rs], out[ts], scale=scale, stream=s, workspace=ws)
            ev = torch.cuda.Event()
            ev.record(s)
            done.append(ev)
        for ev in done:
            main.wait_event(ev)
        return True

    def read_errors(self, clear: bool = True, stream=None) -> int:
        return _lib.cpp_read_device_error(self.dev_err, clear=clear, stream=stream)
