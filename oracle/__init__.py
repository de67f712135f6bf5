"""fp64 CPU oracle for chunked-prefill paged attention (TEST INFRASTRUCTURE).

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline / reference leg of
`bench.py` may import this package. The product library never does, and this
package imports nothing from the product: the two share no code.

Parts:
  attention.c  KV write (bit copy by slot) and paged causal attention, fp64, OpenMP
  split.py     simple and balanced micro-batch split points (pure Python integers)
  planner.py   quadratic latency model, chunk-size solver and post-processing,
               online calibration (windowed two-variable refit)
  scheduler.py token-budget batch builder with page allocation
Parity status of each function (what pins it) is listed in each module's header.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile attention.c into liboracle.so with gcc (-O2, OpenMP, fp64)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _open(path):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.oracle_kv_cache_write.restype = ctypes.c_long
    lib.oracle_kv_cache_write.argtypes = [P, P, P, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_long, P, P]
    lib.oracle_paged_attention.restype = ctypes.c_int
    lib.oracle_paged_attention.argtypes = [P, P, P, P, P, P, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_long,
                                           ctypes.c_double, P, ctypes.c_long, P]
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _open(_LIB)
    return _lib


@contextlib.contextmanager
def using_library(path):
    """Route the oracle's C calls to another build of attention.c while the
    block runs (the mutation test builds copies with planted slips and checks
    that some pin catches each one)."""
    global _lib
    saved = _lib
    _lib = _open(path)
    try:
        yield
    finally:
        _lib = saved


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else ctypes.c_void_p(0)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def kv_cache_write(k, v, slot_mapping, page_size, k_cache, v_cache) -> int:
    """In-place bit copy of k/v rows into the caches at their slots.

    k, v: uint16 [T, Hkv, d]; slot_mapping int64 [T]; caches uint16
    [num_pages, Hkv, P, d]. Returns the number of out-of-range slots skipped."""
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    assert k_cache.dtype == np.uint16 and v_cache.dtype == np.uint16
    T, Hkv, d = k.shape
    assert k_cache.shape[1:] == (Hkv, page_size, d)
    return int(_load().oracle_kv_cache_write(_ptr(k), _ptr(v), _ptr(sm), T, Hkv, d, page_size,
                                              k_cache.shape[0], _ptr(k_cache), _ptr(v_cache)))


def paged_attention(q, k_cache, v_cache, query_lens, seq_lens, block_table, scale=0.0, rows=None):
    """fp64 causal attention of the selected token rows (all rows when None).

    Returns float64 [n_rows, Hq, d]."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k_cache = np.ascontiguousarray(k_cache, dtype=np.uint16)
    v_cache = np.ascontiguousarray(v_cache, dtype=np.uint16)
    ql = np.ascontiguousarray(query_lens, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    T, Hq, d = q.shape
    num_pages, Hkv, P, d2 = k_cache.shape
    assert d2 == d and v_cache.shape == k_cache.shape
    if rows is None:
        rows_arr = None
        n = T
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows_arr.shape[0]
    out = np.zeros((n, Hq, d), dtype=np.float64)
    st = _load().oracle_paged_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(ql), _ptr(sl),
                                        _ptr(bt), bt.shape[0], bt.shape[1], T, Hq, Hkv, d, P,
                                        num_pages, float(scale), _ptr(rows_arr), n, _ptr(out))
    if st != 0:
        raise ValueError(f"oracle_paged_attention: malformed batch (code {st})")
    return out


from .split import simple_split, balanced_split  # noqa: E402,F401
from .planner import (latency_quadratic, target_latency, solve_chunk, postprocess, plan_chunks,  # noqa: E402,F401
                      fit_quadratic, fit_two_var,
                      solve_chunk_two_var, OnlineCalibrator)
from .scheduler import Scheduler  # noqa: E402,F401
