"""The allocation-free attention entry point against the workspace one.

cpp_chunked_prefill_attn_noalloc serves callers that cannot allocate device
memory (a plugin inside a host that owns all device memory, or a C caller with
no allocator of its own): it runs on a scratch area the library keeps in device
global memory. This test calls it twice in a row through the C ABI, on two
different batches (the second finding the first one's data in the scratch
area), and checks each result bit for bit against cpp_chunked_prefill_attn with
a caller workspace (the split partials fit in both, so both make the same
choices), and both against the fp64 oracle within the attention tolerance of
the other tests. A context created through the driver API must get its own
lookup of the scratch area's address (a __device__ array has one address per
context), never the primary context's cached one. The file sorts last so that a
run stopping at the first failure has run everything else.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import bf16_tensor_to_f64, compare, oracle_caches, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _inputs(cpsa, spec):
    import torch
    b = W.make_batch(spec)
    kc = to_dev(W.empty_cache(b).view(np.int16)).view(torch.bfloat16)
    vc = kc.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cpsa.cpp_kv_cache_write(to_dev_bf16(b.hist_k), to_dev_bf16(b.hist_v), to_dev(b.hist_slot_mapping), kc, vc, err)
    cpsa.cpp_kv_cache_write(to_dev_bf16(b.k), to_dev_bf16(b.v), to_dev(b.slot_mapping), kc, vc, err)
    return dict(q=to_dev_bf16(b.q), kc=kc, vc=vc, ql=to_dev(b.query_lens), sl=to_dev(b.seq_lens),
                bt=to_dev(b.block_table), err=err, B=len(spec.qlen), T=b.num_tokens, spec=spec, batch=b)


def _oracle(x):
    b = x["batch"]
    kc, vc = oracle_caches(b)
    return oracle.paged_attention(b.q, kc, vc, b.query_lens, b.seq_lens, b.block_table)


def _with_workspace(cpsa, x):
    import torch
    s = x["spec"]
    ws = torch.empty(cpsa.cpp_attn_workspace_bytes(x["B"], x["T"], s.num_q_heads, s.num_kv_heads, s.head_dim, 8),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty_like(x["q"])
    cpsa.cpp_chunked_prefill_attn(x["q"], x["kc"], x["vc"], x["ql"], x["sl"], x["bt"], out, ws, x["err"],
                                  max_kv_splits=8)
    return out


def _without_workspace(cpsa, x):
    import torch
    out = torch.full_like(x["q"], float("nan"))
    cpsa.cpp_chunked_prefill_attn_noalloc(x["q"], x["kc"], x["vc"], x["ql"], x["sl"], x["bt"], out, x["err"],
                                          max_kv_splits=8)
    return out


def test_noalloc_matches_workspace_entry_point_on_two_calls(cuda_lib):
    import torch
    first = _inputs(cuda_lib, W.BatchSpec(hist=[9000, 300, 5000, 0], qlen=[1, 200, 1, 129], num_q_heads=32,
                                          num_kv_heads=8, head_dim=128, page_size=16, seed=901))
    second = _inputs(cuda_lib, W.BatchSpec(hist=[40, 6000, 1], qlen=[300, 1, 77], num_q_heads=8,
                                           num_kv_heads=2, head_dim=64, page_size=32, seed=902))
    ref1 = _with_workspace(cuda_lib, first)
    ref2 = _with_workspace(cuda_lib, second)
    got1 = _without_workspace(cuda_lib, first)      # first call on this device sets the scratch up
    got2 = _without_workspace(cuda_lib, second)     # second call reuses the scratch the first one left
    torch.cuda.synchronize()
    assert cuda_lib.cpp_read_device_error(first["err"]) == 0
    assert cuda_lib.cpp_read_device_error(second["err"]) == 0
    assert torch.equal(got1.view(torch.int16), ref1.view(torch.int16)), "no-alloc call 1 differs from the workspace call"
    assert torch.equal(got2.view(torch.int16), ref2.view(torch.int16)), "no-alloc call 2 differs from the workspace call"
    for got, x, what in ((got1, first, "call 1"), (got2, second, "call 2")):
        compare(bf16_tensor_to_f64(got), _oracle(x), what=f"no-alloc {what} vs oracle")


def test_noalloc_rejects_a_batch_beyond_the_scratch_area(cuda_lib):
    import torch
    # the work lists alone of 2^24 - 1 requests exceed the 64 MiB scratch area
    need = cuda_lib.cpp_attn_workspace_min_bytes((1 << 24) - 1, 1 << 24, 32, 8, 128, 8)
    assert need > 64 << 20
    q = torch.zeros((1, 32, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 8, 16, 128), dtype=torch.bfloat16, device="cuda")
    ql = torch.zeros((1,), dtype=torch.int32, device="cuda")
    bt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = cuda_lib.load()
    import ctypes
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.cpp_chunked_prefill_attn_noalloc(p(q), p(kc), p(kc), p(ql), p(ql), p(bt), (1 << 24) - 1, 1 << 24, 1,
                                              32, 8, 128, 16, 1, 0.0, 8, p(q), p(err),
                                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == -8     # CPSA_ERR_SCRATCH_TOO_SMALL, nothing launched
    assert lib.cpp_status_string(st).startswith(b"batch needs more")


def test_scratch_address_is_looked_up_per_context(cuda_lib):
    """A second context on the same device, created and made current through
    the driver API, gets the address of its own copy of the scratch area; the
    primary context keeps its cached one. No kernel runs in the second context."""
    import ctypes
    import torch
    torch.zeros(1, device="cuda")                     # the primary context is current
    a_primary = cuda_lib.cpp_noalloc_scratch_address()
    assert a_primary != 0
    assert cuda_lib.cpp_noalloc_scratch_address() == a_primary
    try:
        cu = ctypes.CDLL("libcuda.so.1")
        create, pop, destroy = cu.cuCtxCreate_v2, cu.cuCtxPopCurrent_v2, cu.cuCtxDestroy_v2
    except (OSError, AttributeError):
        pytest.skip("the driver API's context calls are not reachable")
    dev = ctypes.c_int()
    assert cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()) == 0
    ctx = ctypes.c_void_p()
    assert create(ctypes.byref(ctx), 0, dev) == 0      # pushed: current on this thread
    try:
        a_other = cuda_lib.cpp_noalloc_scratch_address()
    finally:
        top = ctypes.c_void_p()
        assert pop(ctypes.byref(top)) == 0 and top.value == ctx.value
        assert destroy(ctx) == 0
    # both arrays are live in one unified address space, so they cannot coincide
    assert a_other != 0 and a_other != a_primary, (hex(a_other), hex(a_primary))
    assert cuda_lib.cpp_noalloc_scratch_address() == a_primary
