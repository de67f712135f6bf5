"""GPU parity of cpp_split_microbatch against the oracle's balanced split (bit-exact)."""
import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


def _gpu_split(cpsa, q, bal, length):
    import torch
    ql = torch.tensor(np.asarray(q, dtype=np.int32), dtype=torch.int32, device="cuda")
    out = torch.full((3,), -7, dtype=torch.int32, device="cuda")
    cpsa.cpp_split_microbatch(ql, out, bal, length)
    b, t, u = out.cpu().tolist()
    return b, t, bool(u)


def _f32(x):
    return float(np.float32(x))   # the kernel receives the threshold as float32


def test_split_hand_cases(cuda_lib):
    assert _gpu_split(cuda_lib, [1, 1, 1, 500, 300], 0.5, 1) == (4, 503, False)
    assert _gpu_split(cuda_lib, [1, 1, 1, 500, 300], 0.7, 1) == (4, 503, True)
    assert _gpu_split(cuda_lib, [7], 0.1, 1) == (0, 0, False)
    assert _gpu_split(cuda_lib, [0, 0], 0.1, 0) == (1, 0, False)
    assert _gpu_split(cuda_lib, [2, 2, 2], 10.0, 0) == (1, 2, True)


def test_split_microbatch_workload(cuda_lib):
    q = W.spec_microbatch().qlen
    assert _gpu_split(cuda_lib, q, 0.1, 256) == oracle.balanced_split(q, _f32(0.1), 256) == (160, 83328, True)


def test_split_random_against_oracle(cuda_lib):
    rng = np.random.default_rng(17)
    for trial in range(200):
        B = int(rng.choice([0, 1, 2, 3, 31, 32, 33, 1023, 1024, 1025, 3000, 5000]))
        q = [int(x) for x in rng.integers(0, 5000, size=B)]
        if trial % 3 == 0:
            q = [1] * int(rng.integers(0, 2000)) + q
        bal = float(rng.choice([0.0, 0.05, 0.1, 0.3, 1.0]))
        length = int(rng.choice([0, 1, 256, 10 ** 6]))
        assert _gpu_split(cuda_lib, q, bal, length) == oracle.balanced_split(q, _f32(bal), length), (trial, B)
