"""ctypes binding of libcpsa.so: argument marshalling only.

Every function here has the name of the C entry point it calls (include/cpsa.h)
and passes torch tensors as raw pointers plus sizes; all computation happens in
the library's CUDA kernels. There is no fallback: when the library is missing
or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcpsa.so")

_lib = None

_c_i64 = ctypes.c_int64
_c_int = ctypes.c_int
_c_p = ctypes.c_void_p
_c_f = ctypes.c_float
_c_d = ctypes.c_double
_c_size = ctypes.c_size_t

# device error bits (mirrors include/cpsa.h)
DEV_SLOT_OUT_OF_RANGE = 0x01
DEV_PAGE_OUT_OF_RANGE = 0x02
DEV_SEQ_LT_QUERY = 0x04
DEV_TOKENS_MISMATCH = 0x08
DEV_SEQ_GT_TABLE = 0x10
DEV_SPLITS_CLAMPED = 0x20
DEV_WAIT_TIMEOUT = 0x40
DEV_PLAN_OVERFLOW = 0x80


class CpsaError(RuntimeError):
    pass


def load():
    """Load libcpsa.so (built in-tree by __graft_entry__.build()); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise CpsaError(f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    lib.cpp_kv_cache_write.restype = _c_int
    lib.cpp_kv_cache_write.argtypes = [_c_p, _c_p, _c_p, _c_i64, _c_int, _c_int, _c_int, _c_i64, _c_p, _c_p, _c_p, _c_p]
    lib.cpp_attn_workspace_bytes.restype = _c_size
    lib.cpp_attn_workspace_bytes.argtypes = [_c_int, _c_i64, _c_int, _c_int, _c_int, _c_int]
    lib.cpp_attn_workspace_min_bytes.restype = _c_size
    lib.cpp_attn_workspace_min_bytes.argtypes = [_c_int, _c_i64, _c_int, _c_int, _c_int, _c_int]
    lib.cpp_chunked_prefill_attn.restype = _c_int
    lib.cpp_chunked_prefill_attn.argtypes = [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_i64, _c_int, _c_int,
                                             _c_int, _c_int, _c_int, _c_i64, _c_f, _c_int, _c_p, _c_p, _c_size,
                                             _c_p, _c_p]
    lib.cpp_chunked_prefill_attn_events.restype = _c_int
    lib.cpp_chunked_prefill_attn_events.argtypes = lib.cpp_chunked_prefill_attn.argtypes + [_c_p]
    lib.cpp_chunked_prefill_attn_write_kv.restype = _c_int
    lib.cpp_chunked_prefill_attn_write_kv.argtypes = [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_int,
                                                      _c_i64, _c_int, _c_int, _c_int, _c_int, _c_int, _c_i64, _c_f,
                                                      _c_int, _c_p, _c_p, _c_size, _c_p, _c_p]
    lib.cpp_chunked_prefill_attn_write_kv_events.restype = _c_int
    lib.cpp_chunked_prefill_attn_write_kv_events.argtypes = lib.cpp_chunked_prefill_attn_write_kv.argtypes + [_c_p]
    lib.cpp_noalloc_scratch_address.restype = _c_int
    lib.cpp_noalloc_scratch_address.argtypes = [ctypes.POINTER(_c_p)]
    lib.cpp_chunked_prefill_attn_noalloc.restype = _c_int
    lib.cpp_chunked_prefill_attn_noalloc.argtypes = [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_i64, _c_int,
                                                     _c_int, _c_int, _c_int, _c_int, _c_i64, _c_f, _c_int, _c_p,
                                                     _c_p, _c_p]
    lib.cpp_split_microbatch.restype = _c_int
    lib.cpp_split_microbatch.argtypes = [_c_p, _c_int, _c_f, ctypes.c_int32, _c_p, _c_p]
    lib.cpp_read_device_error.restype = _c_int
    lib.cpp_read_device_error.argtypes = [_c_p, _c_p, _c_int, _c_p]
    lib.cpp_get_device_error.restype = _c_int
    lib.cpp_get_device_error.argtypes = [_c_p, _c_p, _c_p]
    lib.cpp_plan_chunk_sizes.restype = _c_int
    lib.cpp_plan_chunk_sizes.argtypes = [_c_d, _c_d, _c_d, _c_i64, _c_i64, _c_int, _c_i64, _c_i64, _c_i64, _c_d,
                                         _c_p, _c_i64, _c_p]
    lib.cpp_fit_latency_quadratic.restype = _c_int
    lib.cpp_fit_latency_quadratic.argtypes = [_c_p, _c_p, _c_int, _c_p]
    lib.cpp_fit_latency_two_var.restype = _c_int
    lib.cpp_fit_latency_two_var.argtypes = [_c_p, _c_p, _c_p, _c_p, _c_int, _c_p]
    lib.cpp_online_create.restype = _c_p
    lib.cpp_online_create.argtypes = [_c_d, _c_d, _c_d, _c_i64, _c_int, _c_i64, _c_i64, _c_i64, _c_d, _c_int, _c_int]
    lib.cpp_online_destroy.restype = None
    lib.cpp_online_destroy.argtypes = [_c_p]
    lib.cpp_online_next_chunk.restype = _c_int
    lib.cpp_online_next_chunk.argtypes = [_c_p, _c_i64, _c_i64, _c_p]
    lib.cpp_online_record.restype = _c_int
    lib.cpp_online_record.argtypes = [_c_p, _c_p, _c_p, _c_int, _c_d]
    lib.cpp_online_model.restype = _c_int
    lib.cpp_online_model.argtypes = [_c_p, _c_p, _c_p, _c_p]
    lib.cpp_sched_create.restype = _c_p
    lib.cpp_sched_create.argtypes = [_c_i64, _c_int, _c_i64, _c_p, _c_p, _c_int, _c_int]
    lib.cpp_sched_destroy.restype = None
    lib.cpp_sched_destroy.argtypes = [_c_p]
    lib.cpp_sched_add_request.restype = _c_int
    lib.cpp_sched_add_request.argtypes = [_c_p, _c_i64, _c_i64, _c_i64]
    lib.cpp_sched_step.restype = _c_int
    lib.cpp_sched_step.argtypes = [_c_p, _c_int, _c_i64, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p]
    lib.cpp_sched_commit.restype = _c_int
    lib.cpp_sched_commit.argtypes = [_c_p]
    lib.cpp_sched_stats.restype = _c_int
    lib.cpp_sched_stats.argtypes = [_c_p, _c_p, _c_p, _c_p, _c_p]
    lib.cpp_selftest_exp2.restype = _c_int
    lib.cpp_selftest_exp2.argtypes = [_c_p, _c_p, _c_p, _c_i64, _c_p]
    lib.cpp_selftest_wait_timeout.restype = _c_int
    lib.cpp_selftest_wait_timeout.argtypes = [_c_i64, _c_p, _c_p, _c_p]
    lib.cpp_status_string.restype = ctypes.c_char_p
    lib.cpp_status_string.argtypes = [_c_int]
    _lib = lib
    return lib


def _check(status: int, what: str):
    if status != 0:
        msg = load().cpp_status_string(status).decode()
        raise CpsaError(f"{what} failed: {msg} ({status})")


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return _c_p(stream.cuda_stream)


def _dev(t: torch.Tensor, dtype, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise CpsaError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise CpsaError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise CpsaError(f"{name} must be contiguous")
    return _c_p(t.data_ptr())


def cpp_kv_cache_write(k, v, slot_mapping, k_cache, v_cache, dev_err, stream=None):
    """k, v [T, Hkv, d] bf16; slot_mapping [T] int64; caches [pages, Hkv, P, d] bf16."""
    T, Hkv, d = k.shape
    pages, Hkv2, P, d2 = k_cache.shape
    if v.shape != k.shape or v_cache.shape != k_cache.shape or Hkv2 != Hkv or d2 != d or slot_mapping.shape != (T,):
        raise CpsaError("cpp_kv_cache_write: inconsistent shapes")
    st = load().cpp_kv_cache_write(_dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"),
                                   _dev(slot_mapping, torch.int64, "slot_mapping"), T, Hkv, d, P, pages,
                                   _dev(k_cache, torch.bfloat16, "k_cache"), _dev(v_cache, torch.bfloat16, "v_cache"),
                                   _dev(dev_err, torch.int32, "dev_err"), _stream_ptr(stream))
    _check(st, "cpp_kv_cache_write")


def cpp_attn_workspace_bytes(num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim, max_kv_splits=8):
    n = load().cpp_attn_workspace_bytes(num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim, max_kv_splits)
    if n == 0:
        raise CpsaError("cpp_attn_workspace_bytes: invalid arguments")
    return int(n)


def cpp_attn_workspace_min_bytes(num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim, max_kv_splits=8):
    n = load().cpp_attn_workspace_min_bytes(num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim, max_kv_splits)
    if n == 0:
        raise CpsaError("cpp_attn_workspace_min_bytes: invalid arguments")
    return int(n)


def cpp_chunked_prefill_attn(q, k_cache, v_cache, query_lens, seq_lens, block_table, out, workspace, dev_err,
                             scale=0.0, max_kv_splits=8, stream=None):
    """q/out [T, Hq, d] bf16; caches [pages, Hkv, P, d] bf16; lens [B] int32; block_table [B, M] int32;
    workspace uint8 of cpp_attn_workspace_*_bytes; dev_err int32 [1] (bit flags)."""
    T, Hq, d = q.shape
    pages, Hkv, P, d2 = k_cache.shape
    B = query_lens.shape[0]
    if out.shape != q.shape or v_cache.shape != k_cache.shape or d2 != d or seq_lens.shape != (B,) \
            or block_table.dim() != 2 or block_table.shape[0] != B:
        raise CpsaError("cpp_chunked_prefill_attn: inconsistent shapes")
    st = load().cpp_chunked_prefill_attn(
        _dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.bfloat16, "k_cache"),
        _dev(v_cache, torch.bfloat16, "v_cache"), _dev(query_lens, torch.int32, "query_lens"),
        _dev(seq_lens, torch.int32, "seq_lens"), _dev(block_table, torch.int32, "block_table"),
        B, T, block_table.shape[1], Hq, Hkv, d, P, pages, float(scale), int(max_kv_splits),
        _dev(out, torch.bfloat16, "out"), _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
        _dev(dev_err, torch.int32, "dev_err"), _stream_ptr(stream))
    _check(st, "cpp_chunked_prefill_attn")


def cpp_chunked_prefill_attn_events(q, k_cache, v_cache, query_lens, seq_lens, block_table, out, workspace,
                                    dev_err, events, scale=0.0, max_kv_splits=8, stream=None):
    """cpp_chunked_prefill_attn recording 5 torch.cuda.Event marks (None allowed) around its kernels."""
    T, Hq, d = q.shape
    pages, Hkv, P, d2 = k_cache.shape
    B = query_lens.shape[0]
    if out.shape != q.shape or v_cache.shape != k_cache.shape or d2 != d or seq_lens.shape != (B,) \
            or block_table.dim() != 2 or block_table.shape[0] != B or len(events) != 5:
        raise CpsaError("cpp_chunked_prefill_attn_events: inconsistent shapes")
    for e in events:
        if e is not None and not e.cuda_event:
            e.record(stream)          # torch creates its events lazily, on first record
    evs = (_c_p * 5)(*[_c_p(e.cuda_event) if e is not None else _c_p(0) for e in events])
    st = load().cpp_chunked_prefill_attn_events(
        _dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.bfloat16, "k_cache"),
        _dev(v_cache, torch.bfloat16, "v_cache"), _dev(query_lens, torch.int32, "query_lens"),
        _dev(seq_lens, torch.int32, "seq_lens"), _dev(block_table, torch.int32, "block_table"),
        B, T, block_table.shape[1], Hq, Hkv, d, P, pages, float(scale), int(max_kv_splits),
        _dev(out, torch.bfloat16, "out"), _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
        _dev(dev_err, torch.int32, "dev_err"), _stream_ptr(stream), evs)
    _check(st, "cpp_chunked_prefill_attn_events")


def cpp_chunked_prefill_attn_write_kv(q, k, v, slot_mapping, k_cache, v_cache, query_lens, seq_lens, block_table,
                                      out, workspace, dev_err, scale=0.0, max_kv_splits=8, stream=None,
                                      events=None):
    """KV write fused into the attention: k, v [T, Hkv, d] bf16 and slot_mapping [T] int64 as for
    cpp_kv_cache_write (the caches are written), the rest as for cpp_chunked_prefill_attn.
    events: None, or 5 torch.cuda.Event marks (None allowed) as for cpp_chunked_prefill_attn_events."""
    T, Hq, d = q.shape
    pages, Hkv, P, d2 = k_cache.shape
    B = query_lens.shape[0]
    if out.shape != q.shape or v_cache.shape != k_cache.shape or d2 != d or seq_lens.shape != (B,) \
            or block_table.dim() != 2 or block_table.shape[0] != B or k.shape != (T, Hkv, d) \
            or v.shape != k.shape or slot_mapping.shape != (T,):
        raise CpsaError("cpp_chunked_prefill_attn_write_kv: inconsistent shapes")
    args = (_dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"),
            _dev(slot_mapping, torch.int64, "slot_mapping"), _dev(k_cache, torch.bfloat16, "k_cache"),
            _dev(v_cache, torch.bfloat16, "v_cache"), _dev(query_lens, torch.int32, "query_lens"),
            _dev(seq_lens, torch.int32, "seq_lens"), _dev(block_table, torch.int32, "block_table"),
            B, T, block_table.shape[1], Hq, Hkv, d, P, pages, float(scale), int(max_kv_splits),
            _dev(out, torch.bfloat16, "out"), _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
            _dev(dev_err, torch.int32, "dev_err"), _stream_ptr(stream))
    if events is None:
        st = load().cpp_chunked_prefill_attn_write_kv(*args)
    else:
        if len(events) != 5:
            raise CpsaError("cpp_chunked_prefill_attn_write_kv: events must hold 5 entries")
        for e in events:
            if e is not None and not e.cuda_event:
                e.record(stream)          # torch creates its events lazily, on first record
        evs = (_c_p * 5)(*[_c_p(e.cuda_event) if e is not None else _c_p(0) for e in events])
        st = load().cpp_chunked_prefill_attn_write_kv_events(*args, evs)
    _check(st, "cpp_chunked_prefill_attn_write_kv")


def cpp_noalloc_scratch_address():
    """Device address (int) of the no-alloc scratch area in the current CUDA context."""
    addr = _c_p()
    _check(load().cpp_noalloc_scratch_address(ctypes.byref(addr)), "cpp_noalloc_scratch_address")
    return int(addr.value or 0)


def cpp_chunked_prefill_attn_noalloc(q, k_cache, v_cache, query_lens, seq_lens, block_table, out, dev_err,
                                     scale=0.0, max_kv_splits=8, stream=None):
    """cpp_chunked_prefill_attn without a workspace: for callers that cannot
    allocate device memory, the library's own fixed scratch area is used (see
    include/cpsa.h: calls that overlap on the GPU must not share it)."""
    T, Hq, d = q.shape
    pages, Hkv, P, d2 = k_cache.shape
    B = query_lens.shape[0]
    if out.shape != q.shape or v_cache.shape != k_cache.shape or d2 != d or seq_lens.shape != (B,) \
            or block_table.dim() != 2 or block_table.shape[0] != B:
        raise CpsaError("cpp_chunked_prefill_attn_noalloc: inconsistent shapes")
    st = load().cpp_chunked_prefill_attn_noalloc(
        _dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.bfloat16, "k_cache"),
        _dev(v_cache, torch.bfloat16, "v_cache"), _dev(query_lens, torch.int32, "query_lens"),
        _dev(seq_lens, torch.int32, "seq_lens"), _dev(block_table, torch.int32, "block_table"),
        B, T, block_table.shape[1], Hq, Hkv, d, P, pages, float(scale), int(max_kv_splits),
        _dev(out, torch.bfloat16, "out"), _dev(dev_err, torch.int32, "dev_err"), _stream_ptr(stream))
    _check(st, "cpp_chunked_prefill_attn_noalloc")


def cpp_split_microbatch(query_lens, out3, balance_threshold=0.1, length_threshold=256, stream=None):
    """Writes (batch_split, token_split, use_two) into the int32 [3] device tensor out3."""
    st = load().cpp_split_microbatch(_dev(query_lens, torch.int32, "query_lens"), query_lens.shape[0],
                                     float(balance_threshold), int(length_threshold),
                                     _dev(out3, torch.int32, "out3"), _stream_ptr(stream))
    _check(st, "cpp_split_microbatch")


def cpp_read_device_error(dev_err, clear=True, stream=None) -> int:
    host = ctypes.c_uint32(0)
    st = load().cpp_read_device_error(_dev(dev_err, torch.int32, "dev_err"), ctypes.byref(host), int(clear),
                                      _stream_ptr(stream))
    _check(st, "cpp_read_device_error")
    return int(host.value)


def cpp_get_device_error(dev_err, stream=None) -> int:
    """The device error word, left as it is (reading it synchronises the stream)."""
    host = ctypes.c_uint32(0)
    st = load().cpp_get_device_error(_dev(dev_err, torch.int32, "dev_err"), ctypes.byref(host), _stream_ptr(stream))
    _check(st, "cpp_get_device_error")
    return int(host.value)


def cpp_plan_chunk_sizes(a, b, c, prompt_len, base_chunk_size, page_size, min_chunk=64, max_model_len=0,
                         max_num_scheduled_tokens=0, smooth_factor=1.0):
    lib = load()
    n = ctypes.c_int64(0)
    # caps (max_model_len - L, max_num_scheduled_tokens) may cut chunks below
    # min_chunk, down to one token: a prompt has at most prompt_len chunks
    cap = max(16, int(prompt_len) + 1)
    buf = (ctypes.c_int64 * cap)()
    st = lib.cpp_plan_chunk_sizes(a, b, c, prompt_len, base_chunk_size, page_size, min_chunk, max_model_len,
                                  max_num_scheduled_tokens, smooth_factor, buf, cap, ctypes.byref(n))
    _check(st, "cpp_plan_chunk_sizes")
    return [int(buf[i]) for i in range(n.value)]


def _dbl(xs):
    arr = (ctypes.c_double * len(xs))(*[float(x) for x in xs])
    return arr


def cpp_fit_latency_quadratic(lengths, times):
    coef = (ctypes.c_double * 3)()
    _check(load().cpp_fit_latency_quadratic(_dbl(lengths), _dbl(times), len(lengths), coef),
           "cpp_fit_latency_quadratic")
    return [coef[0], coef[1], coef[2]]


def cpp_fit_latency_two_var(x0, x1, x2, times):
    coef = (ctypes.c_double * 3)()
    _check(load().cpp_fit_latency_two_var(_dbl(x0), _dbl(x1), _dbl(x2), _dbl(times), len(times), coef),
           "cpp_fit_latency_two_var")
    return [coef[0], coef[1], coef[2]]


class OnlineChunker:
    """Handle of the library's online chunk-size controller (cpp_online_* in cpsa.h)."""

    def __init__(self, a, b, c, base_chunk_size, page_size, min_chunk=64, max_model_len=0,
                 max_num_scheduled_tokens=0, smooth_factor=1.0, window=30, min_points=5):
        self._lib = load()
        self._h = self._lib.cpp_online_create(a, b, c, base_chunk_size, page_size, min_chunk, max_model_len,
                                              max_num_scheduled_tokens, smooth_factor, window, min_points)
        if not self._h:
            raise CpsaError("cpp_online_create: invalid arguments")

    def next_chunk(self, history, remaining) -> int:
        out = ctypes.c_int64(0)
        _check(self._lib.cpp_online_next_chunk(self._h, history, remaining, ctypes.byref(out)),
               "cpp_online_next_chunk")
        return int(out.value)

    def record(self, chunks, histories, time_ms):
        cs = (ctypes.c_int64 * len(chunks))(*[int(x) for x in chunks])
        hs = (ctypes.c_int64 * len(histories))(*[int(x) for x in histories])
        _check(self._lib.cpp_online_record(self._h, cs, hs, len(chunks), float(time_ms)), "cpp_online_record")

    def model(self):
        """((a, b, c), batches recorded, calibrated)."""
        coef = (ctypes.c_double * 3)()
        n, cal = ctypes.c_int(0), ctypes.c_int(0)
        _check(self._lib.cpp_online_model(self._h, coef, ctypes.byref(n), ctypes.byref(cal)), "cpp_online_model")
        return (coef[0], coef[1], coef[2]), n.value, bool(cal.value)

    def close(self):
        if getattr(self, "_h", None):
            self._lib.cpp_online_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()


class BatchScheduler:
    """Handle of the library's token-budget batch builder (cpp_sched_* in cpsa.h).
    step() returns the batch's host arrays (numpy); commit() applies it."""

    def __init__(self, token_budget, page_size, num_pages, page_order=None, chunk_caps=(), tile_align=0,
                 max_reqs=4096, max_blocks=4096):
        import numpy as np
        self._np = np
        self._lib = load()
        order = None
        if page_order is not None:
            self._order = np.ascontiguousarray(np.asarray(page_order, dtype=np.int32))
            order = self._order.ctypes.data_as(_c_p)
        caps = (ctypes.c_int64 * max(1, len(chunk_caps)))(*[int(c) for c in chunk_caps])
        self._h = self._lib.cpp_sched_create(token_budget, page_size, num_pages, order, caps, len(chunk_caps),
                                             tile_align)
        if not self._h:
            raise CpsaError("cpp_sched_create: invalid arguments")
        self.max_reqs, self.max_blocks, self.max_tokens = max_reqs, max_blocks, token_budget

    def add_request(self, rid, prompt_len, max_new_tokens):
        _check(self._lib.cpp_sched_add_request(self._h, rid, prompt_len, max_new_tokens), "cpp_sched_add_request")

    def step(self):
        np = self._np
        ids = np.zeros(self.max_reqs, np.int64)
        ql = np.zeros(self.max_reqs, np.int32)
        sl = np.zeros(self.max_reqs, np.int32)
        bt = np.zeros((self.max_reqs, self.max_blocks), np.int32)
        sm = np.zeros(max(1, self.max_tokens), np.int64)
        nr, nt = ctypes.c_int(0), ctypes.c_int64(0)
        p = lambda a: a.ctypes.data_as(_c_p)
        _check(self._lib.cpp_sched_step(self._h, self.max_reqs, self.max_tokens, self.max_blocks, p(ids), p(ql),
                                        p(sl), p(bt), p(sm), ctypes.byref(nr), ctypes.byref(nt)), "cpp_sched_step")
        B, T = nr.value, nt.value
        return {"req_ids": ids[:B].copy(), "query_lens": ql[:B].copy(), "seq_lens": sl[:B].copy(),
                "block_table": bt[:B].copy(), "slot_mapping": sm[:T].copy()}

    def commit(self):
        _check(self._lib.cpp_sched_commit(self._h), "cpp_sched_commit")

    def stats(self):
        """(waiting, running, finished, free pages)."""
        v = [ctypes.c_int64(0) for _ in range(4)]
        _check(self._lib.cpp_sched_stats(self._h, *[ctypes.byref(x) for x in v]), "cpp_sched_stats")
        return tuple(x.value for x in v)

    def close(self):
        if getattr(self, "_h", None):
            self._lib.cpp_sched_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()


def cpp_selftest_exp2(x, stream=None):
    """(poly, hw) = the attention kernels' FMA-pipe and hardware exp2 of the float32 CUDA tensor x."""
    poly = torch.empty_like(x)
    hw = torch.empty_like(x)
    _check(load().cpp_selftest_exp2(_dev(x, torch.float32, "x"), _dev(poly, torch.float32, "poly"),
                                    _dev(hw, torch.float32, "hw"), x.numel(), _stream_ptr(stream)),
           "cpp_selftest_exp2")
    return poly, hw


def cpp_selftest_wait_timeout(limit_ns, dev_err, stream=None):
    """Runs the bounded-wait self-test; returns the int32 [3] device tensor
    (warp 0 wait ok, warp 1 wait ok, microseconds warp 1 waited)."""
    out = torch.full((3,), -1, dtype=torch.int32, device=dev_err.device)
    _check(load().cpp_selftest_wait_timeout(int(limit_ns), _dev(dev_err, torch.int32, "dev_err"),
                                            _dev(out, torch.int32, "out3"), _stream_ptr(stream)),
           "cpp_selftest_wait_timeout")
    return out
