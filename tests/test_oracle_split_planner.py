"""Pins of the oracle's micro-batch split and chunk planner (CPU only)."""
import math

import numpy as np
import pytest

import oracle
import workloads as W


def brute_force_split(q, balance, length):
    B = len(q)
    if B < 2:
        return 0, 0, False
    total = sum(q)
    cands = [(abs(sum(q[:k]) - total // 2), k) for k in range(1, B)]
    _, k = min(cands)                      # min on (distance, k): smallest k on ties
    n1 = sum(q[:k]); n2 = total - n1
    if min(n1, n2) == 0:
        return k, n1, False
    return k, n1, (abs(n1 - n2) / min(n1, n2) <= balance) and min(n1, n2) >= length


def test_balanced_split_hand_case():
    q = [1, 1, 1, 500, 300]
    assert oracle.balanced_split(q, 0.5, 1) == (4, 503, False)    # imbalance 203/300 = 0.677
    assert oracle.balanced_split(q, 0.7, 1) == (4, 503, True)
    assert oracle.balanced_split(q, 0.7, 301) == (4, 503, False)  # 300 < length threshold


def test_simple_split_hand_case():
    assert oracle.simple_split([1, 1, 1, 500, 300]) == (2, 2)


def test_microbatch_workload_split():
    spec = W.spec_microbatch()
    assert sum(spec.qlen) == 166528
    assert oracle.balanced_split(spec.qlen, 0.1, 256) == (160, 83328, True)


def test_degenerate_splits():
    assert oracle.balanced_split([], 0.1, 1) == (0, 0, False)
    assert oracle.balanced_split([7], 0.1, 1) == (0, 0, False)
    assert oracle.balanced_split([0, 0], 0.1, 0) == (1, 0, False)
    assert oracle.balanced_split([3, 3], 0.0, 3) == (1, 3, True)
    # ties: cumulative 2 and 4 are equally far from best = 3 -> smaller k
    assert oracle.balanced_split([2, 2, 2], 10.0, 0) == (1, 2, True)


def test_balanced_split_matches_brute_force():
    rng = np.random.default_rng(7)
    for _ in range(400):
        B = int(rng.integers(0, 40))
        q = [int(x) for x in rng.integers(0, 3000, size=B)]
        if rng.random() < 0.3:
            q = [1] * int(rng.integers(0, 20)) + q
        bal = float(rng.choice([0.0, 0.05, 0.1, 0.5, 2.0]))
        length = int(rng.choice([0, 1, 256, 4096]))
        assert oracle.balanced_split(q, bal, length) == brute_force_split(q, bal, length)


def test_solver_root_at_zero_history_is_base():
    for a, b in [(1e-6, 2e-3), (3.3e-7, 0.01), (1e-9, 1e-1), (2.0, 5.0)]:
        T = oracle.target_latency(a, b, 0.4, 4096)
        x = oracle.solve_chunk(0, a, b, T, 4096)
        assert abs(x - 4096) <= 4096 * 1e-12
        assert oracle.postprocess(x, 0, 4096, 128) == 4096


def test_solver_equalises_latency_before_rounding():
    a, b, c = 2.5e-7, 3e-3, 0.7
    T = oracle.target_latency(a, b, c, 4096)
    for L in [0, 1, 100, 4096, 10000, 32000, 10 ** 6]:
        x = oracle.solve_chunk(L, a, b, T, 4096)
        gain = oracle.latency_quadratic(L + x, a, b, c) - oracle.latency_quadratic(L, a, b, c)
        assert abs(gain - T) <= 1e-9 * T
        assert 0 < x <= 4096 + 1e-9


def test_solver_matches_printed_root_where_it_is_stable():
    a, b = 1e-3, 2.0
    T = oracle.target_latency(a, b, 0.0, 512)
    for L in [0, 10, 300]:
        lin = 2 * a * L + b
        printed = (-lin + math.sqrt(lin * lin + 4 * a * T)) / (2 * a)
        assert abs(oracle.solve_chunk(L, a, b, T, 512) - printed) <= 1e-9 * printed


def test_solver_linear_fallbacks():
    assert oracle.solve_chunk(100, 0.0, 2.0, 10.0, 4096) == 5.0
    assert oracle.solve_chunk(100, -1.0, 0.0, 10.0, 4096) == 4096.0


def test_postprocess_rounding_and_caps():
    assert oracle.postprocess(1000.0, 0, 4096, 128) == 896
    assert oracle.postprocess(100.0, 0, 4096, 128) == 64          # minimum 64
    assert oracle.postprocess(40.0, 0, 4096, 16) == 64
    assert oracle.postprocess(1000.0, 0, 4096, 16) == 992
    assert oracle.postprocess(1000.0, 32000, 4096, 128, max_model_len=32768) == 768
    assert oracle.postprocess(1000.0, 0, 4096, 128, max_num_scheduled_tokens=512) == 512
    assert oracle.postprocess(1000.0, 0, 4096, 128, smooth_factor=0.5) == 2432   # (1000+4096)/2 = 2548


def test_plan_covers_prompt_and_shrinks():
    a, b, c = 2.5e-7, 3e-3, 0.7
    chunks = oracle.plan_chunks(32768, a, b, c, 4096, 128)
    assert sum(chunks) == 32768
    assert chunks[0] == 4096
    assert all(x >= y for x, y in zip(chunks[:-2], chunks[1:-1]))   # non-increasing but the remainder
    assert all(x % 128 == 0 or x == 64 for x in chunks[:-1])


def test_fits_recover_exact_coefficients():
    l = np.array(W.chunk_profile_sizes(4096, 64), dtype=np.float64)
    assert l[0] == 64 and l[-1] == 4096 and len(l) == 64
    coef, res = oracle.fit_quadratic(l, 3e-7 * l * l + 2e-3 * l + 0.5)
    np.testing.assert_allclose(coef, [3e-7, 2e-3, 0.5], rtol=1e-8)
    C = [[512]] * 10 + [[64, 128], [1024]]
    H = [[512 * i] for i in range(10)] + [[0, 64], [0]]
    t = [sum(1e-7 * c * (c + h) + 1e-3 * (c + h) + 0.25 for c, h in zip(cs, hs)) for cs, hs in zip(C, H)]
    coef2, _ = oracle.fit_two_var(C, H, t)
    np.testing.assert_allclose(coef2, [1e-7, 1e-3, 0.25], rtol=1e-7)


# ------------------------------------------------------------ online calibration
def f_two_var(C, H, a, b, c):
    return a * C * (C + H) + b * (C + H) + c


def test_calibrated_root_at_zero_history_is_base():
    a, b = 3e-7, 2e-3
    base = 4096
    T = a * base * base + b * base
    assert abs(oracle.solve_chunk_two_var(0, a, b, T, base) - base) < 1e-9 * base


def test_calibrated_root_equalises_chunk_time():
    """f(C, H) - f(0, H) = T at the unrounded root, for many (a, b, H)."""
    rng = np.random.default_rng(11)
    for _ in range(200):
        a, b = rng.uniform(1e-9, 1e-6), rng.uniform(1e-5, 1e-2)
        H = float(rng.integers(0, 200000))
        T = a * 4096 ** 2 + b * 4096
        C = oracle.solve_chunk_two_var(H, a, b, T, 4096)
        lhs = f_two_var(C, H, a, b, 0.3) - f_two_var(0.0, H, a, b, 0.3)
        assert abs(lhs - T) <= 1e-9 * T
        assert 0 < C <= 4096 + 1e-6     # history only makes chunks smaller
    assert oracle.solve_chunk_two_var(5000, 0.0, 2e-3, 8.0, 4096) == pytest.approx(4000.0)
    assert oracle.solve_chunk_two_var(5000, 0.0, 0.0, 8.0, 4096) == 4096.0


def test_online_calibration_recovers_the_model_and_forgets_old_batches():
    true_a, b0, c0 = (2e-7, 1.5e-3, 0.4)
    cal = oracle.OnlineCalibrator(1e-7, 1e-3, 0.1, 4096, 128, window=6, min_points=5)
    L = 0
    for i in range(4):                          # startup model until the 5th batch
        x = cal.next_chunk(L, 32768 - L)
        cal.record([x], [L], f_two_var(x, L, true_a, b0, c0))
        L += x
        assert not cal.calibrated and cal.coef == [1e-7, 1e-3, 0.1]
    x = cal.next_chunk(L, 32768 - L)
    cal.record([x], [L], f_two_var(x, L, true_a, b0, c0))
    assert cal.calibrated
    np.testing.assert_allclose(cal.coef, [true_a, b0, c0], rtol=1e-6)
    # the machine slows down: after `window` batches of the new model only it is recovered exactly
    new = (3e-7, 2e-3, 0.6)
    for i in range(6):
        C, H = 256 + 128 * i, 1000 * i
        cal.record([C, 64], [H, 0], f_two_var(C, H, *new) + f_two_var(64, 0, *new))   # c once per chunk
    np.testing.assert_allclose(cal.coef, list(new), rtol=1e-6)


def test_online_controller_matches_oracle():
    """The library's controller (host C++) against the oracle's, on a noisy latency
    model: identical chunk sizes, coefficients to 1e-9."""
    import chunked_prefill_paged_slot_gb300 as cpsa
    rng = np.random.default_rng(5)
    for window, smooth in ((30, 1.0), (8, 0.7)):
        ours = cpsa.OnlineChunker(2e-7, 1e-3, 0.2, 4096, 128, window=window, smooth_factor=smooth)
        ref = oracle.OnlineCalibrator(2e-7, 1e-3, 0.2, 4096, 128, window=window, smooth_factor=smooth)
        L, prompt = 0, 65536
        while L < prompt:
            x1, x2 = ours.next_chunk(L, prompt - L), ref.next_chunk(L, prompt - L)
            assert x1 == x2, (L, x1, x2)
            t = f_two_var(x1, L, 3e-7, 2.2e-3, 0.35) * (1.0 + 0.03 * rng.standard_normal())
            ours.record([x1], [L], t)
            ref.record([x1], [L], t)
            L += x1
        coef, n, cal = ours.model()
        assert cal and ref.calibrated and n == len(ref.times)
        np.testing.assert_allclose(coef, ref.coef, rtol=1e-9)
        ours.close()
