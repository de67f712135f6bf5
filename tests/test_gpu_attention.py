"""GPU parity of cpp_chunked_prefill_attn against the fp64 oracle.

Every batch here is small enough for the oracle to compute every row; the
caches start as NaN patterns, so a kernel that touches an unwritten slot
without masking it produces NaN and fails. Bound: max-abs 2e-2 and relative
Frobenius 5e-3 (bf16 inputs, fp32 accumulation, bf16 P and output)."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import bf16_tensor_to_f64, compare, oracle_caches, run_gpu_batch, run_gpu_batch_fused, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def check(cpsa, spec, max_kv_splits=8, workspace_bytes=None, scale=0.0, expect_flags=0):
    b = W.make_batch(spec)
    got, flags, _, _ = run_gpu_batch(cpsa, b, max_kv_splits=max_kv_splits, workspace_bytes=workspace_bytes,
                                     scale=scale)
    assert flags == expect_flags, f"device flags {flags:#x}"
    kc, vc = oracle_caches(b)
    ref = oracle.paged_attention(b.q, kc, vc, b.query_lens, b.seq_lens, b.block_table, scale=scale)
    return compare(got, ref, what=spec.name or str(spec.qlen))


def test_small_chunk_workload(cuda_lib):
    """History 256 + chunk 128, 4/4 heads, d=64, page 16."""
    check(cuda_lib, W.spec_one_chunk_small())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (32, 8), (6, 2), (16, 1)])
def test_heads_and_dims(cuda_lib, d, hq, hkv):
    spec = W.BatchSpec(hist=[130, 0, 7], qlen=[200, 129, 1], num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                       page_size=16, seed=100 + hq + d)
    check(cuda_lib, spec)


@pytest.mark.parametrize("P", [8, 16, 32, 64, 128, 256])
def test_page_sizes(cuda_lib, P):
    spec = W.BatchSpec(hist=[300, 1000, 0], qlen=[77, 1, 260], num_q_heads=8, num_kv_heads=2, head_dim=128,
                       page_size=P, seed=200 + P, extra_pages=5)
    check(cuda_lib, spec)


def test_ragged_mixed_batch(cuda_lib):
    """Decode rows first, then chunks with ragged tails, a zero-length request inside."""
    spec = W.BatchSpec(hist=[900, 33, 4000, 0, 511, 512, 513, 0, 77],
                       qlen=[1, 1, 1, 2, 128, 127, 129, 0, 383],
                       num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16, seed=300)
    check(cuda_lib, spec)


@pytest.mark.parametrize("splits", [1, 2, 8])
def test_long_history_splits(cuda_lib, splits):
    """Long histories: prefill tiles past 32 KV tiles and decode rows past 4096 keys split."""
    spec = W.BatchSpec(hist=[9000, 5000, 6000], qlen=[1, 150, 1], num_q_heads=8, num_kv_heads=2,
                       head_dim=128, page_size=16, seed=400 + splits)
    check(cuda_lib, spec, max_kv_splits=splits)


def test_workspace_clamp_still_correct(cuda_lib):
    spec = W.BatchSpec(hist=[9000, 5000], qlen=[1, 150], num_q_heads=8, num_kv_heads=2, head_dim=128,
                       page_size=16, seed=450)
    minb = cuda_lib.cpp_attn_workspace_min_bytes(2, 151, 8, 2, 128, 8)
    check(cuda_lib, spec, max_kv_splits=8, workspace_bytes=minb, expect_flags=cuda_lib.DEV_SPLITS_CLAMPED)


def test_custom_scale(cuda_lib):
    spec = W.BatchSpec(hist=[64], qlen=[64], num_q_heads=4, num_kv_heads=2, head_dim=64, page_size=16, seed=500)
    check(cuda_lib, spec, scale=0.3)


def test_decode_only_batch(cuda_lib):
    rng = np.random.default_rng(3)
    ctx = [int(x) for x in rng.integers(1, 3000, size=40)]
    spec = W.BatchSpec(hist=[c - 1 for c in ctx], qlen=[1] * 40, num_q_heads=32, num_kv_heads=8, head_dim=128,
                       page_size=16, seed=501)
    check(cuda_lib, spec)


def test_tiny_prefills(cuda_lib):
    spec = W.BatchSpec(hist=[0, 1, 2, 15, 16, 17], qlen=[2, 2, 3, 1, 5, 16], num_q_heads=4, num_kv_heads=1,
                       head_dim=64, page_size=8, seed=502)
    check(cuda_lib, spec)


def test_device_errors_are_flagged_not_faulted(cuda_lib):
    import torch
    spec = W.BatchSpec(hist=[10, 20], qlen=[5, 1], num_q_heads=4, num_kv_heads=2, head_dim=64, page_size=16,
                       seed=503)
    b = W.make_batch(spec)
    # seq_len < query_len on request 0
    bad = W.make_batch(spec)
    bad.seq_lens = bad.seq_lens.copy()
    bad.seq_lens[0] = 2
    _, flags, _, _ = run_gpu_batch(cuda_lib, bad)
    assert flags & cuda_lib.DEV_SEQ_LT_QUERY
    # a block_table entry past the pool
    bt = b.block_table.copy()
    bt[1, 0] = b.num_pages + 5
    _, flags, _, _ = run_gpu_batch(cuda_lib, b, block_table=bt)
    assert flags & cuda_lib.DEV_PAGE_OUT_OF_RANGE
    # sum(query_lens) != num_tokens
    mm = W.make_batch(spec)
    mm.query_lens = np.array([4, 1], dtype=np.int32)
    _, flags, _, _ = run_gpu_batch(cuda_lib, mm)
    assert flags & cuda_lib.DEV_TOKENS_MISMATCH
    torch.cuda.synchronize()


def test_host_argument_errors(cuda_lib):
    import torch
    q = torch.zeros((4, 4, 96), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((2, 2, 16, 96), dtype=torch.bfloat16, device="cuda")
    ql = torch.tensor([4], dtype=torch.int32, device="cuda")
    bt = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(cuda_lib.CpsaError):    # head_dim 96 unsupported
        cuda_lib.cpp_chunked_prefill_attn(q, kc, kc.clone(), ql, ql.clone(), bt, q.clone(), ws, e)
    q = torch.zeros((4, 4, 64), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((2, 2, 12, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cuda_lib.CpsaError):    # page size 12 unsupported
        cuda_lib.cpp_chunked_prefill_attn(q, kc, kc.clone(), ql, ql.clone(), bt, q.clone(), ws, e)
    kc = torch.zeros((2, 2, 16, 64), dtype=torch.bfloat16, device="cuda")
    tiny = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(cuda_lib.CpsaError):    # workspace too small
        cuda_lib.cpp_chunked_prefill_attn(q, kc, kc.clone(), ql, ql.clone(), bt, q.clone(), tiny, e)
    assert cuda_lib.cpp_read_device_error(e) == 0


def test_get_device_error_reads_without_clearing(cuda_lib):
    """cpp_get_device_error returns the word and leaves it; cpp_read_device_error clears it."""
    import torch
    k = torch.zeros((2, 2, 64), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 2, 16, 64), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    slots = torch.tensor([3, 16], dtype=torch.int64, device="cuda")   # 16 = past the one 16-slot page
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cuda_lib.cpp_kv_cache_write(k, k, slots, kc, vc, err)
    assert cuda_lib.cpp_get_device_error(err) == cuda_lib.DEV_SLOT_OUT_OF_RANGE
    assert cuda_lib.cpp_get_device_error(err) == cuda_lib.DEV_SLOT_OUT_OF_RANGE
    assert cuda_lib.cpp_read_device_error(err, clear=True) == cuda_lib.DEV_SLOT_OUT_OF_RANGE
    assert cuda_lib.cpp_get_device_error(err) == 0


def test_events_entry_point_on_a_mixed_batch(cuda_lib):
    """cpp_chunked_prefill_attn_events (plain stream order, events between the kernels)
    on decode rows plus prefills with split units: same result as the oracle."""
    import torch
    spec = W.BatchSpec(hist=[5000, 0, 300, 7000, 64], qlen=[1, 400, 1, 257, 1], num_q_heads=32, num_kv_heads=8,
                       head_dim=128, page_size=16, seed=611)
    b = W.make_batch(spec)

    kc = to_dev(W.empty_cache(b).view(np.int16)).view(torch.bfloat16)
    vc = kc.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cuda_lib.cpp_kv_cache_write(to_dev_bf16(b.hist_k), to_dev_bf16(b.hist_v), to_dev(b.hist_slot_mapping), kc, vc, err)
    cuda_lib.cpp_kv_cache_write(to_dev_bf16(b.k), to_dev_bf16(b.v), to_dev(b.slot_mapping), kc, vc, err)
    B, T = len(spec.qlen), b.num_tokens
    ws = torch.empty(cuda_lib.cpp_attn_workspace_bytes(B, T, 32, 8, 128, 8), dtype=torch.uint8, device="cuda")
    out = torch.full((T, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    cuda_lib.cpp_chunked_prefill_attn_events(to_dev_bf16(b.q), kc, vc, to_dev(b.query_lens), to_dev(b.seq_lens),
                                             to_dev(b.block_table), out, ws, err, ev, max_kv_splits=8)
    torch.cuda.synchronize()
    assert cuda_lib.cpp_read_device_error(err) == 0
    assert all(ev[i].elapsed_time(ev[i + 1]) >= 0 for i in range(4))
    okc, okv = oracle_caches(b)
    ref = oracle.paged_attention(b.q, okc, okv, b.query_lens, b.seq_lens, b.block_table)
    compare(bf16_tensor_to_f64(out), ref, what="events entry point")


def test_split_merges_are_repeatable_bit_for_bit(cuda_lib):
    """Units cut into 2 to 10+ pieces: whichever piece finishes last merges (at the
    end of a CTA's run through shared memory, else from L2), and the merge sums in
    piece order with the merging piece's own O rounded as it would have been
    stored, so repeated calls give identical bits; the output matches the oracle."""
    spec = W.BatchSpec(hist=[3000, 700, 12000, 64, 0], qlen=[300, 256, 40, 2, 600], num_q_heads=32,
                       num_kv_heads=8, head_dim=128, page_size=16, seed=510)
    b = W.make_batch(spec)
    runs = [run_gpu_batch(cuda_lib, b)[0] for _ in range(4)]
    runs += [run_gpu_batch_fused(cuda_lib, b)[0] for _ in range(4)]
    for r in runs[1:4]:
        assert np.array_equal(runs[0].view(np.uint64), r.view(np.uint64))
    for r in runs[5:]:
        assert np.array_equal(runs[4].view(np.uint64), r.view(np.uint64))
    kc, vc = oracle_caches(b)
    ref = oracle.paged_attention(b.q, kc, vc, b.query_lens, b.seq_lens, b.block_table)
    compare(runs[0], ref, what="split merges")
    compare(runs[4], ref, what="split merges, fused")


@pytest.mark.parametrize("fused", [False, True])
def test_short_histories_keep_units_whole(cuda_lib, fused):
    """When every unit is at least a stream-K run long and the longest is within
    a cut's cost of it, the plan keeps units whole, one per CTA (a 512-token chunk
    at history 512; two such requests side by side): every row against the oracle."""
    for hist, qlen, seed in (([512], [512], 520), ([512, 640], [512, 384], 521)):
        spec = W.BatchSpec(hist=hist, qlen=qlen, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=128,
                           seed=seed)
        b = W.make_batch(spec)
        got = (run_gpu_batch_fused if fused else run_gpu_batch)(cuda_lib, b)[0]
        kc, vc = oracle_caches(b)
        ref = oracle.paged_attention(b.q, kc, vc, b.query_lens, b.seq_lens, b.block_table)
        compare(got, ref, what=f"whole units {hist}")


@pytest.mark.parametrize("fused", [False, True])
def test_few_long_requests_take_the_block_plan(cuda_lib, fused):
    """At most 32 requests but more than 8192 tokens also take the block-wide plan
    kernel (a warp per request): three prompts and a decode row, 8301 tokens,
    sampled rows of every request (its first and last rows, tile edges) against
    the oracle."""
    spec = W.BatchSpec(hist=[0, 1000, 3000, 500], qlen=[3000, 2600, 1, 2700], num_q_heads=32, num_kv_heads=8,
                       head_dim=128, page_size=16, seed=540 + int(fused))
    b = W.make_batch(spec)
    got, flags, _, _ = (run_gpu_batch_fused if fused else run_gpu_batch)(cuda_lib, b)
    assert flags == 0, f"device flags {flags:#x}"
    starts = np.concatenate([[0], np.cumsum(spec.qlen)])
    rng = np.random.default_rng(541)
    rows = [0, 127, 128, 2999, 3000, 3127, 3128, 5599, 5600, 5601, 5728, 8300]
    rows = np.unique(np.concatenate([rows, rng.choice(int(starts[-1]), 40, replace=False)]))
    kc, vc = oracle_caches(b)
    ref = oracle.paged_attention(b.q, kc, vc, b.query_lens, b.seq_lens, b.block_table, rows=rows)
    compare(got[rows], ref, what="few long requests" + (" fused" if fused else ""))


def test_whole_units_in_the_block_plan(cuda_lib):
    """More than 32 requests take the block-wide plan kernel; 40 requests of 128
    rows at history 1024 (one kv head, one q-head pair) give 40 units of 9 tiles
    against runs of 4, so units stay whole there too: every row against the oracle."""
    spec = W.BatchSpec(hist=[1024] * 40, qlen=[128] * 40, num_q_heads=2, num_kv_heads=1, head_dim=64,
                       page_size=64, seed=530)
    check(cuda_lib, spec)
