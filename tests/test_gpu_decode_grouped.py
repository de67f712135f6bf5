"""GPU parity of the grouped decode kernel: decode rows whose kv heads come in
groups of 8 (or 4) are attended by items that cover a whole group, each stage
reading every head of a page with one TMA box. Checked against the fp64 oracle
on every row, with the KV write as its own call and fused into the attention
call (the row's own key patched into the stage and stored to its slot), across
page sizes, head dims, q heads per kv head up to 16, and long contexts whose
rows are split along keys and merged by the combine kernel."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import cache_bits, compare, oracle_caches, run_gpu_batch, run_gpu_batch_fused

pytestmark = pytest.mark.gpu


def _check(cpsa, spec, max_kv_splits=8, fused=False):
    b = W.make_batch(spec)
    run = run_gpu_batch_fused if fused else run_gpu_batch
    got, flags, kc, vc = run(cpsa, b, max_kv_splits=max_kv_splits)
    assert flags == 0, hex(flags)
    okc, ovc = oracle_caches(b)
    if fused:
        assert np.array_equal(cache_bits(kc), okc) and np.array_equal(cache_bits(vc), ovc), "cache contents"
    ref = oracle.paged_attention(b.q, okc, ovc, b.query_lens, b.seq_lens, b.block_table)
    compare(got, ref, what=f"{spec.qlen[:4]} P={spec.page_size} fused={fused}")


def _decode_spec(n, hq, hkv, d, page, seed, lo=1, hi=3000, prefill=None):
    rng = np.random.default_rng(seed)
    ctx = [int(x) for x in rng.integers(lo, hi, size=n)]
    hist = [c - 1 for c in ctx]
    qlen = [1] * n
    if prefill is not None:
        hist.append(prefill[0])
        qlen.append(prefill[1])
    return W.BatchSpec(hist=hist, qlen=qlen, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, page_size=page,
                       seed=seed)


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("page", [8, 16, 32, 256])
def test_grouped_page_sizes(cuda_lib, page, fused):
    """8 kv heads per item; page 8 takes two boxes per stage, larger pages one box
    of 16 rows at an offset inside the page."""
    _check(cuda_lib, _decode_spec(24, 32, 8, 128, page, 2000 + page + int(fused)), fused=fused)


@pytest.mark.parametrize("hq,hkv,d", [(16, 4, 128), (64, 4, 128), (64, 8, 64), (32, 16, 128), (8, 8, 64)])
def test_grouped_heads_and_dims(cuda_lib, hq, hkv, d):
    """Groups of 4 and 8 heads, 16 q heads per kv head (both mma row halves),
    head_dim 64, two groups per row (16 kv heads), one q head per kv head."""
    for fused in (False, True):
        _check(cuda_lib, _decode_spec(20, hq, hkv, d, 16, 2100 + hq + hkv + d), fused=fused)


@pytest.mark.parametrize("splits", [1, 2, 8])
def test_grouped_long_contexts_split(cuda_lib, splits):
    """Contexts past 4096 keys split along keys (fp32 partials, combine kernel), beside a prefill."""
    spec = _decode_spec(12, 32, 8, 128, 16, 2200 + splits, lo=3000, hi=14000, prefill=(700, 300))
    _check(cuda_lib, spec, max_kv_splits=splits)
    _check(cuda_lib, spec, max_kv_splits=splits, fused=True)


def test_grouped_ragged_contexts(cuda_lib):
    """Contexts of 1, 15, 16, 17 and 8191 keys: stages that end inside a page and a box."""
    spec = W.BatchSpec(hist=[0, 14, 15, 16, 8190, 31, 32], qlen=[1] * 7, num_q_heads=32, num_kv_heads=8,
                       head_dim=128, page_size=16, seed=2300)
    _check(cuda_lib, spec)
    _check(cuda_lib, spec, fused=True)


def test_per_head_kernel_still_serves_other_head_counts(cuda_lib):
    """2 kv heads (neither a group of 8 nor of 4): the per-head decode kernel."""
    _check(cuda_lib, _decode_spec(20, 8, 2, 128, 16, 2400))
    _check(cuda_lib, _decode_spec(20, 6, 2, 64, 32, 2401), fused=True)
