"""The library's own chunk planner and latency fits (host C++ in libcpsa.so)
against the oracle's, directly (CPU only).

The planner follows the vllm-ascend "Dynamic Chunked Pipeline Parallel (CPP)"
design page, "runtime phase: dynamic prediction" (next chunk from
f(L + x) - f(L) = T, then smoothing, page alignment, minimum and caps); the fits
follow its "startup phase: profiling" (f(l) = a l^2 + b l + c) and "online
calibration" (f(C, H) = a C (C + H) + b (C + H) + c) sections. The chunk lists
must be identical integer lists; the fitted coefficients agree to 1e-9 of their
scale (the library solves the normal equations, the oracle calls lstsq)."""
import itertools

import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def cpsa():
    from chunked_prefill_paged_slot_gb300 import build as b
    b.build()
    import chunked_prefill_paged_slot_gb300 as lib
    lib.load()
    return lib


# (a, b, c) of latency models in ms: GB300-sized ones, a linear one, a <= 0 and b <= 0 fallbacks
MODELS = [(4.75e-9, 3.87e-5, 0.024), (2e-7, 1e-3, 0.2), (1e-6, 0.0, 0.05), (0.0, 2e-4, 0.01),
          (-3e-9, 5e-5, 0.02), (0.0, 0.0, 0.3), (-1e-8, -1e-4, 0.1), (3e-8, -1e-5, 0.02)]


def test_plan_chunk_sizes_grid(cpsa):
    """Every combination of model, prompt, base, page, smoothing, minimum and caps:
    the library's list equals the oracle's, element for element."""
    n = 0
    for (a, b, c), prompt, base, page, smooth, min_chunk, caps in itertools.product(
            MODELS, (32768, 5000, 777), (512, 4096), (16, 128), (1.0, 0.7, 0.3), (64, 256),
            ((0, 0), (40000, 0), (0, 1024), (36000, 2048))):
        mml, mst = caps
        ours = cpsa.cpp_plan_chunk_sizes(a, b, c, prompt, base, page, min_chunk, mml, mst, smooth)
        ref = oracle.plan_chunks(prompt, a, b, c, base, page, smooth_factor=smooth, min_chunk=min_chunk,
                                 max_model_len=mml or None, max_num_scheduled_tokens=mst or None)
        assert ours == ref, ((a, b, c), prompt, base, page, smooth, min_chunk, caps)
        assert sum(ours) == prompt
        n += 1
    assert n == len(MODELS) * 3 * 2 * 2 * 3 * 2 * 4


def test_plan_chunk_sizes_model_len_cap_below_prompt(cpsa):
    """max_model_len below the prompt: the cap max_model_len - L reaches zero and every
    later chunk is one token (both sides clamp to at least 1)."""
    for a, b, c in MODELS[:3]:
        ours = cpsa.cpp_plan_chunk_sizes(a, b, c, 700, 256, 16, 64, 600, 0, 1.0)
        ref = oracle.plan_chunks(700, a, b, c, 256, 16, max_model_len=600)
        assert ours == ref and sum(ours) == 700


def _rel_close(x, y, tol=1e-9):
    x, y = np.asarray(x, np.float64), np.asarray(y, np.float64)
    scale = np.maximum(np.abs(y), 1e-300)
    assert np.all(np.abs(x - y) <= tol * scale), (x, y)


def test_fit_quadratic_matches_oracle(cpsa):
    """Noisy samples of f(l) at the 64 profile sizes base*i/64 (and at random sizes)."""
    rng = np.random.default_rng(12)
    for a, b, c in MODELS[:4]:
        for sizes in (np.arange(1, 65) * 64.0, np.sort(rng.integers(16, 8192, size=40)).astype(np.float64)):
            t = (a * sizes ** 2 + b * sizes + c) * (1.0 + 0.05 * rng.standard_normal(sizes.size)) + 1e-3
            ours = cpsa.cpp_fit_latency_quadratic(sizes.tolist(), t.tolist())
            ref, _ = oracle.fit_quadratic(sizes, t)
            _rel_close(ours, ref)
            # and the fitted curves agree at every sample
            X = np.stack([sizes ** 2, sizes, np.ones_like(sizes)], 1)
            np.testing.assert_allclose(X @ np.asarray(ours), X @ ref, rtol=1e-10, atol=0)


def test_fit_two_var_matches_oracle(cpsa):
    """Noisy batches of one to three chunks at assorted histories: features
    [sum C (C + H), sum (C + H), N] built by the oracle's own fit, handed to the
    library's fit as columns."""
    rng = np.random.default_rng(13)
    for a, b, c in ((3e-7, 2.2e-3, 0.35), (4.75e-9, 3.87e-5, 0.024)):
        chunks, hists, times = [], [], []
        for _ in range(45):
            k = int(rng.integers(1, 4))
            cs = rng.integers(64, 4096, size=k)
            hs = rng.integers(0, 32768, size=k)
            chunks.append(cs)
            hists.append(hs)
            f = float(np.sum(a * cs * (cs + hs) + b * (cs + hs) + c))
            times.append(f * (1.0 + 0.03 * rng.standard_normal()))
        ref, _ = oracle.fit_two_var(chunks, hists, times)
        x0 = [float(np.sum(cs * (cs + hs))) for cs, hs in zip(chunks, hists)]
        x1 = [float(np.sum(cs + hs)) for cs, hs in zip(chunks, hists)]
        x2 = [float(len(cs)) for cs in chunks]
        ours = cpsa.cpp_fit_latency_two_var(x0, x1, x2, times)
        _rel_close(ours, ref)


def test_fits_recover_exact_models(cpsa):
    """Noise-free samples: both fits return the generating coefficients."""
    l = np.arange(1, 65) * 64.0
    ours = cpsa.cpp_fit_latency_quadratic(l.tolist(), (2e-7 * l * l + 1e-3 * l + 0.2).tolist())
    np.testing.assert_allclose(ours, [2e-7, 1e-3, 0.2], rtol=1e-9)
    C = np.array([512.0, 1024, 2048, 256, 4096])
    H = np.array([0.0, 512, 8192, 30000, 100])
    t = 3e-7 * C * (C + H) + 2e-3 * (C + H) + 0.5
    ours = cpsa.cpp_fit_latency_two_var((C * (C + H)).tolist(), (C + H).tolist(), [1.0] * 5, t.tolist())
    np.testing.assert_allclose(ours, [3e-7, 2e-3, 0.5], rtol=1e-9)
