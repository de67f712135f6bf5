"""The attention kernels' base-2 exponentials against fp64 2**x: the FMA-pipe
polynomial (Cody-Waite range reduction + degree-3 minimax, relative error bound
7.5e-5 from its fit, plus fp32 rounding) and the hardware ex2.approx."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_fma_pipe_exp2_within_its_error_bound(cuda_lib):
    import torch
    rng = np.random.default_rng(0)
    x = np.concatenate([np.linspace(-125.0, 127.0, 200001), rng.uniform(-30, 9, 200000),
                        np.arange(-125, 128, dtype=np.float64),              # exact integers
                        np.arange(-125, 127) + 0.5,                          # rounding ties
                        [0.0, -0.0, 1e-30, -1e-30]]).astype(np.float32)
    poly, hw = cuda_lib.cpp_selftest_exp2(torch.from_numpy(x).cuda())
    poly = poly.cpu().numpy().astype(np.float64)
    hw = hw.cpu().numpy().astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel_poly = np.abs(poly / ref - 1.0)
    rel_hw = np.abs(hw / ref - 1.0)
    assert np.all(np.isfinite(poly))
    assert rel_poly.max() <= 7.5e-5 + 2e-7, rel_poly.max()
    assert rel_hw.max() <= 1e-6, rel_hw.max()


def test_fma_pipe_exp2_clamps_outside_its_range(cuda_lib):
    import torch
    x = torch.tensor([-1000.0, -126.0, -float("inf"), 200.0], device="cuda")
    poly, hw = cuda_lib.cpp_selftest_exp2(x)
    poly = poly.cpu().numpy()
    assert np.all(poly[:3] > 0) and np.all(poly[:3] < 1e-37)     # 2^-125 at most: negligible beside p >= 1
    assert np.isclose(poly[3], 2.0 ** 127, rtol=1e-4)
    assert hw.cpu().numpy()[2] == 0.0
