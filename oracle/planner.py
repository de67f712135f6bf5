"""Dynamic chunk-size planner (TEST INFRASTRUCTURE).

Follows the vllm-ascend design page "dynamic-chunk pipeline parallel (CPP)",
sections "quadratic latency model", "runtime phase: dynamic prediction" and
"online calibration":

* latency model f(l) = a*l^2 + b*l + c;
* target T = f(base_chunk_size) - f(0);
* next chunk x solves f(L + x) - f(L) = T, i.e. a*x^2 + (2aL + b)*x - T = 0,
  whose positive root is the quadratic formula's "+" branch;
* post-processing: blend with base_chunk_size by smooth_factor, round down to a
  multiple of page_size (at least 64), cap at max_model_len - L and at
  max_num_scheduled_tokens;
* two-variable model f(C, H) = a*C*(C+H) + b*(C+H) + c with features
  [sum (C+H)*C, sum (C+H), N] per batch.

Readings where the page is silent or numerically fragile:
  * the root is evaluated as 2T / ((2aL+b) + sqrt((2aL+b)^2 + 4aT)), the same
    root without the cancellation of the printed form at large L;
    a <= 0 falls back to the linear root T / b, and b <= 0 as well to base;
  * smoothing is x_s = s*x + (1-s)*base (the page gives no formula);
  * rounding down to the page multiple allows a relative slack of 1e-9, so a
    root that is a page multiple in exact arithmetic is not lost to rounding;
  * the last chunk of a prompt is whatever remains.

Online calibration (same page, "online calibration"): after every batch the
features [sum C(C+H), sum (C+H), N] and the measured time are recorded; once
enough batches are in (the page: 5 to 30 points) the two-variable model is
refitted by least squares, here over a sliding window of the last `window`
batches. Readings:
  * with the two-variable model the next chunk C at history H solves
    f(C, H) - f(0, H) = T, i.e. a*C^2 + (a*H + b)*C - T = 0 (the counterpart of
    f(L + x) - f(L) = T; f(0, H) = b*H + c is what a batch costs at that history
    before any new token);
  * T = f(base, 0) - f(0, 0) = a*base^2 + b*base is recomputed from the current
    model, the page's definition of the target applied to the calibrated model;
  * until the first refit the startup model and its solver are used.

Pinned by closed forms: x(L=0) = base, f(L+x) - f(L) = T before rounding, the
rounding/cap rules, least-squares fits that recover exact coefficients, the
calibrated root at H = 0 equal to base, and a window that forgets older batches.
The fits are numpy.linalg.lstsq (a library routine).
"""
from __future__ import annotations

import math

import numpy as np


def latency_quadratic(l, a, b, c):
    return a * l * l + b * l + c


def target_latency(a, b, c, base_chunk_size):
    return latency_quadratic(base_chunk_size, a, b, c) - latency_quadratic(0, a, b, c)


def solve_chunk(L, a, b, T, base_chunk_size):
    """Unrounded root x of a*x^2 + (2aL+b)*x - T = 0 (positive branch)."""
    if a <= 0.0:
        if b <= 0.0:
            return float(base_chunk_size)
        return T / b
    lin = 2.0 * a * L + b
    disc = lin * lin + 4.0 * a * T
    return 2.0 * T / (lin + math.sqrt(disc))


def postprocess(x, L, base_chunk_size, page_size, smooth_factor=1.0, min_chunk=64,
                max_model_len=None, max_num_scheduled_tokens=None):
    xs = smooth_factor * x + (1.0 - smooth_factor) * base_chunk_size
    units = math.floor(xs / page_size * (1.0 + 1e-9))
    aligned = max(min_chunk, units * page_size)
    if max_model_len is not None:
        aligned = min(aligned, max_model_len - L)
    if max_num_scheduled_tokens is not None:
        aligned = min(aligned, max_num_scheduled_tokens)
    return int(aligned)


def plan_chunks(prompt_len, a, b, c, base_chunk_size, page_size, smooth_factor=1.0,
                min_chunk=64, max_model_len=None, max_num_scheduled_tokens=None):
    """Chunk sizes covering prompt_len tokens, each solved at its own prefix L."""
    T = target_latency(a, b, c, base_chunk_size)
    chunks = []
    L = 0
    while L < prompt_len:
        x = solve_chunk(L, a, b, T, base_chunk_size)
        n = postprocess(x, L, base_chunk_size, page_size, smooth_factor, min_chunk,
                        max_model_len, max_num_scheduled_tokens)
        n = max(1, min(n, prompt_len - L))
        chunks.append(n)
        L += n
    return chunks


def fit_quadratic(lengths, times):
    """Least-squares (a, b, c) of f(l) = a*l^2 + b*l + c; returns (coef, residuals)."""
    l = np.asarray(lengths, dtype=np.float64)
    t = np.asarray(times, dtype=np.float64)
    X = np.stack([l * l, l, np.ones_like(l)], axis=1)
    coef, *_ = np.linalg.lstsq(X, t, rcond=None)
    return coef, t - X @ coef


def fit_two_var(chunks, histories, times):
    """Least-squares (a, b, c) of f(C, H) = a*C*(C+H) + b*(C+H) + c.

    Each sample is one batch; chunks/histories are per-sample lists (a batch may
    hold several chunks), giving the features [sum C*(C+H), sum (C+H), N]."""
    rows = []
    for cs, hs in zip(chunks, histories):
        cs = np.atleast_1d(np.asarray(cs, dtype=np.float64))
        hs = np.atleast_1d(np.asarray(hs, dtype=np.float64))
        rows.append([float(np.sum(cs * (cs + hs))), float(np.sum(cs + hs)), float(len(cs))])
    X = np.asarray(rows)
    t = np.asarray(times, dtype=np.float64)
    coef, *_ = np.linalg.lstsq(X, t, rcond=None)
    return coef, t - X @ coef


def solve_chunk_two_var(H, a, b, T, base_chunk_size):
    """Unrounded root C of a*C^2 + (a*H + b)*C - T = 0 (f(C, H) - f(0, H) = T)."""
    if a <= 0.0:
        if b <= 0.0:
            return float(base_chunk_size)
        return T / b
    lin = a * H + b
    return 2.0 * T / (lin + math.sqrt(lin * lin + 4.0 * a * T))


class OnlineCalibrator:
    """The online chunk-size controller, step by step as the page describes it."""

    def __init__(self, a, b, c, base_chunk_size, page_size, min_chunk=64, max_model_len=None,
                 max_num_scheduled_tokens=None, smooth_factor=1.0, window=30, min_points=5):
        self.coef = [float(a), float(b), float(c)]
        self.calibrated = False
        self.base, self.page = base_chunk_size, page_size
        self.min_chunk, self.max_model_len = min_chunk, max_model_len
        self.max_sched, self.smooth = max_num_scheduled_tokens, smooth_factor
        self.window, self.min_points = window, min_points
        self.rows, self.times = [], []

    def next_chunk(self, history, remaining):
        a, b, c = self.coef
        T = a * self.base * self.base + b * self.base
        if self.calibrated:
            x = solve_chunk_two_var(history, a, b, T, self.base)
        else:
            x = solve_chunk(history, a, b, T, self.base)
        n = postprocess(x, history, self.base, self.page, self.smooth, self.min_chunk,
                        self.max_model_len, self.max_sched)
        return max(1, min(n, remaining))

    def record(self, chunks, histories, time_ms):
        cs = np.atleast_1d(np.asarray(chunks, dtype=np.float64))
        hs = np.atleast_1d(np.asarray(histories, dtype=np.float64))
        self.rows.append([float(np.sum(cs * (cs + hs))), float(np.sum(cs + hs)), float(len(cs))])
        self.times.append(float(time_ms))
        if len(self.times) >= self.min_points:
            X = np.asarray(self.rows[-self.window:])
            t = np.asarray(self.times[-self.window:])
            if np.linalg.matrix_rank(X) == 3:
                coef, *_ = np.linalg.lstsq(X, t, rcond=None)
                self.coef = [float(v) for v in coef]
                self.calibrated = True
