"""GPU parity on seeded random batches against the fp64 oracle, every row.

Each case draws a mixed batch -- up to a dozen requests, each a decode row or a
prefill chunk with a random history and length, zero-length requests among
them -- with a random head layout, page size and KV-split limit, and runs it
with the KV write as its own call and fused into the attention call (then the
caches are also checked bit for bit against the oracle's KV write). The work
split, which piece of a unit each CTA holds, which warp merges, which epilogue
path a unit's rows take, all follow from the batch, so random batches reach
combinations the hand-written cases do not. Sizes stay small enough for the
oracle to compute every row. A second set draws larger batches (up to 32
requests, prompts up to 3000 tokens, often past 8192 tokens in all, which the
block-wide plan kernel lays out) and checks every decode row and sampled rows
of every prompt (its first and last, its tile edges, a few more)."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import cache_bits, compare, oracle_caches, run_gpu_batch, run_gpu_batch_fused

pytestmark = pytest.mark.gpu

HEADS = [(32, 8, 128), (8, 2, 64), (16, 4, 128), (6, 2, 128), (8, 8, 64)]


def _spec(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 13))
    hist, qlen = [], []
    for _ in range(n):
        kind = rng.random()
        if kind < 0.35:
            qlen.append(1)
            hist.append(int(rng.integers(0, 3000)))
        elif kind < 0.42:
            qlen.append(0)
            hist.append(int(rng.integers(0, 500)))
        else:
            qlen.append(int(rng.integers(2, 700)))
            hist.append(int(rng.choice([0, int(rng.integers(1, 3000))])))
    hq, hkv, d = HEADS[int(rng.integers(len(HEADS)))]
    page = int(rng.choice([8, 16, 32, 128]))
    return W.BatchSpec(hist=hist, qlen=qlen, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, page_size=page,
                       seed=seed, extra_pages=int(rng.integers(0, 4))), int(rng.choice([1, 2, 8]))


@pytest.mark.parametrize("seed", list(range(4000, 4016)))
def test_random_batch(cuda_lib, seed):
    spec, splits = _spec(seed)
    if sum(spec.qlen) == 0:
        pytest.skip("no tokens drawn")
    b = W.make_batch(spec)
    kc, vc = oracle_caches(b)
    ref = oracle.paged_attention(b.q, kc, vc, b.query_lens, b.seq_lens, b.block_table)
    what = f"seed {seed}: qlen {spec.qlen} hist {spec.hist} P={spec.page_size} splits={splits}"
    got, flags, _, _ = run_gpu_batch(cuda_lib, b, max_kv_splits=splits)
    assert flags == 0, f"{what}: device flags {flags:#x}"
    compare(got, ref, what=what)
    got_f, flags_f, kc_f, vc_f = run_gpu_batch_fused(cuda_lib, b, max_kv_splits=splits)
    assert flags_f == 0, f"{what} (fused): device flags {flags_f:#x}"
    assert np.array_equal(cache_bits(kc_f), kc) and np.array_equal(cache_bits(vc_f), vc), f"{what}: caches"
    compare(got_f, ref, what=what + " (fused)")


def _large_spec(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(2, 33))
    hist, qlen = [], []
    for _ in range(n):
        if rng.random() < 0.5:
            qlen.append(1)
            hist.append(int(rng.integers(0, 6000)))
        else:
            qlen.append(int(rng.integers(2, 3001)))
            hist.append(int(rng.choice([0, int(rng.integers(1, 5000))])))
    hq, hkv, d = HEADS[int(rng.integers(len(HEADS)))]
    page = int(rng.choice([16, 32, 128]))
    return W.BatchSpec(hist=hist, qlen=qlen, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, page_size=page,
                       seed=seed), int(rng.choice([2, 8]))


def _sample_rows(spec, rng):
    rows, t = [], 0
    for q in spec.qlen:
        if q == 1:
            rows.append(t)
        elif q > 1:
            edges = [x for k in range(128, q, 128) for x in (k - 1, k)]
            pick = rng.choice(q, min(q, 4), replace=False).tolist()
            rows += [t + x for x in [0, q - 1] + edges[:6] + pick]
        t += q
    return np.unique(np.asarray(rows, dtype=np.int64))


@pytest.mark.parametrize("seed", list(range(4100, 4112)))
def test_random_large_batch_sampled_rows(cuda_lib, seed):
    spec, splits = _large_spec(seed)
    b = W.make_batch(spec)
    rows = _sample_rows(spec, np.random.default_rng(seed))
    kc, vc = oracle_caches(b)
    ref = oracle.paged_attention(b.q, kc, vc, b.query_lens, b.seq_lens, b.block_table, rows=rows)
    what = f"seed {seed}: {len(spec.qlen)} requests, {sum(spec.qlen)} tokens, P={spec.page_size} splits={splits}"
    got, flags, _, _ = run_gpu_batch(cuda_lib, b, max_kv_splits=splits)
    assert flags == 0, f"{what}: device flags {flags:#x}"
    compare(got[rows], ref, what=what)
    got_f, flags_f, kc_f, vc_f = run_gpu_batch_fused(cuda_lib, b, max_kv_splits=splits)
    assert flags_f == 0, f"{what} (fused): device flags {flags_f:#x}"
    assert np.array_equal(cache_bits(kc_f), kc) and np.array_equal(cache_bits(vc_f), vc), f"{what}: caches"
    compare(got_f[rows], ref, what=what + " (fused)")
