"""Failure detection on the GPU without a fault: the bounded waits of the
kernels run out on a barrier that nothing arrives at, report
CPSA_DEV_WAIT_TIMEOUT through the device error word, and the abort flag stops a
second role of the CTA long before its own (one-second) limit; the context stays
usable (an attention call right after matches the oracle)."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import bf16_tensor_to_f64, compare, oracle_caches, run_gpu_batch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_us", [50, 2000])
def test_wait_runs_out_and_aborts_the_other_role(cuda_lib, limit_us):
    import torch
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = cuda_lib.cpp_selftest_wait_timeout(limit_us * 1000, err)
    torch.cuda.synchronize()
    a_ok, b_ok, b_us = (int(x) for x in out.cpu().tolist())
    assert a_ok == 0 and b_ok == 0, (a_ok, b_ok)
    # the sleeping role left on the abort flag, not on its own one-second limit
    assert b_us < 500_000, b_us
    assert b_us >= limit_us // 2, b_us
    flags = cuda_lib.cpp_read_device_error(err)
    assert flags == cuda_lib.DEV_WAIT_TIMEOUT, hex(flags)


def test_context_usable_after_a_timeout(cuda_lib):
    import torch
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cuda_lib.cpp_selftest_wait_timeout(20_000, err)
    torch.cuda.synchronize()
    assert cuda_lib.cpp_read_device_error(err) == cuda_lib.DEV_WAIT_TIMEOUT
    b = W.make_batch(W.BatchSpec(hist=[300, 1000], qlen=[130, 1], num_q_heads=8, num_kv_heads=2, head_dim=128,
                                 page_size=16, seed=71))
    got, flags, _, _ = run_gpu_batch(cuda_lib, b)
    assert flags == 0
    kc, vc = oracle_caches(b)
    compare(got, oracle.paged_attention(b.q, kc, vc, b.query_lens, b.seq_lens, b.block_table),
            what="attention after a timeout")


def test_limit_outside_range_is_refused(cuda_lib):
    import torch
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = cuda_lib.load()
    import ctypes
    out = torch.zeros(3, dtype=torch.int32, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for bad in (0, 999, 100_000_001):
        assert lib.cpp_selftest_wait_timeout(bad, ctypes.c_void_p(err.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                             s) == -2
