"""GPU parity of the self-planned chunk kernel: a batch of one prefill request
skips the plan kernel, and every chunk-kernel CTA computes its own stream-K run
(units, run length and cut rule of the plan; split units' partial rows and merge
counters addressed by the run they start in; epoch-tagged merge counters that
no kernel clears between calls). Each case is checked against the fp64 oracle.
Batches of one request up to 6656 tokens (32 q / 8 kv heads on 152 SMs, each
unit weighted by its fixed cost of two tiles) take this path; 6784 tokens takes
the plan kernel and is checked beside it."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import (bf16_tensor_to_f64, compare, oracle_caches, run_gpu_batch, run_gpu_batch_fused, to_dev,
                     to_dev_bf16)

pytestmark = pytest.mark.gpu


def _oracle_rows(b, rows=None):
    kc, vc = oracle_caches(b)
    return oracle.paged_attention(b.q, kc, vc, b.query_lens, b.seq_lens, b.block_table, rows=rows)


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("hist,q", [(9000, 512), (0, 512), (512, 512), (300, 1000), (127, 129), (5, 2)])
def test_single_prefill(cuda_lib, fused, hist, q):
    """Long histories (units cut across runs and merged), no history (short units,
    many per run), units kept whole, ragged tails, a two-token prompt."""
    spec = W.BatchSpec(hist=[hist], qlen=[q], num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                       seed=1100 + hist + q + int(fused))
    b = W.make_batch(spec)
    run = run_gpu_batch_fused if fused else run_gpu_batch
    got, flags, _, _ = run(cuda_lib, b)
    assert flags == 0, hex(flags)
    compare(got, _oracle_rows(b), what=f"h={hist} q={q}" + (" fused" if fused else ""))


@pytest.mark.parametrize("d,hq,hkv", [(64, 8, 8), (128, 6, 2), (64, 16, 1), (128, 4, 4)])
def test_single_prefill_heads(cuda_lib, d, hq, hkv):
    """One q head per CTA (odd groups) and head pairs; head_dim 64 and 128."""
    spec = W.BatchSpec(hist=[2000], qlen=[300], num_q_heads=hq, num_kv_heads=hkv, head_dim=d, page_size=32,
                       seed=1200 + d + hq + hkv)
    b = W.make_batch(spec)
    for run in (run_gpu_batch, run_gpu_batch_fused):
        got, flags, _, _ = run(cuda_lib, b)
        assert flags == 0, hex(flags)
        compare(got, _oracle_rows(b), what=f"d={d} {hq}/{hkv}")


@pytest.mark.parametrize("q", [3968, 6656, 6784])
def test_size_on_either_side_of_the_self_plan_bound(cuda_lib, q):
    """6656 tokens: self-planned (the most pieces a run may hold); 6784: the plan
    kernel; 3968 as well. Sampled rows, every tile edge."""
    spec = W.BatchSpec(hist=[300], qlen=[q], num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                       seed=1300 + q)
    b = W.make_batch(spec)
    rng = np.random.default_rng(q)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, q - 129, q - 128, q - 1], rng.choice(q, 40, replace=False)]))
    for run in (run_gpu_batch, run_gpu_batch_fused):
        got, flags, _, _ = run(cuda_lib, b)
        assert flags == 0, hex(flags)
        compare(got[rows], _oracle_rows(b, rows=rows), what=f"q={q}")


def test_clamped_partials_run_without_cuts(cuda_lib):
    """A workspace without room for split partials: units are not cut, the call
    says so with CPSA_DEV_SPLITS_CLAMPED, and the result is still exact."""
    spec = W.BatchSpec(hist=[9000], qlen=[384], num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                       seed=1400)
    b = W.make_batch(spec)
    ws = cuda_lib.cpp_attn_workspace_min_bytes(1, 384, 32, 8, 128, 8)
    got, flags, _, _ = run_gpu_batch(cuda_lib, b, workspace_bytes=ws)
    assert flags == cuda_lib.DEV_SPLITS_CLAMPED, hex(flags)
    compare(got, _oracle_rows(b), what="clamped")
    got1, flags1, _, _ = run_gpu_batch(cuda_lib, b, max_kv_splits=1)
    assert flags1 == 0
    compare(got1, _oracle_rows(b), what="max_kv_splits 1")


def test_one_workspace_many_calls(cuda_lib):
    """Calls of changing lengths on one workspace: each finds the merge counters of
    the one before (another epoch) and must not take them for its own."""
    import torch
    cases = [(9000, 512), (9000, 512), (3000, 200), (12000, 1000), (0, 512), (9000, 512), (700, 64)]
    ws = torch.empty(cuda_lib.cpp_attn_workspace_bytes(1, 1000, 32, 8, 128, 8), dtype=torch.uint8, device="cuda")
    for i, (hist, q) in enumerate(cases):
        b = W.make_batch(W.BatchSpec(hist=[hist], qlen=[q], num_q_heads=32, num_kv_heads=8, head_dim=128,
                                     page_size=16, seed=1500 + i))
        s = b.spec
        kc = to_dev(W.empty_cache(b).view(np.int16)).view(torch.bfloat16)
        vc = kc.clone()
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        cuda_lib.cpp_kv_cache_write(to_dev_bf16(b.hist_k), to_dev_bf16(b.hist_v), to_dev(b.hist_slot_mapping), kc,
                                    vc, err)
        cuda_lib.cpp_kv_cache_write(to_dev_bf16(b.k), to_dev_bf16(b.v), to_dev(b.slot_mapping), kc, vc, err)
        out = torch.empty((q, 32, 128), dtype=torch.bfloat16, device="cuda")
        cuda_lib.cpp_chunked_prefill_attn(to_dev_bf16(b.q), kc, vc, to_dev(b.query_lens), to_dev(b.seq_lens),
                                          to_dev(b.block_table), out, ws, err, max_kv_splits=8)
        torch.cuda.synchronize()
        assert cuda_lib.cpp_read_device_error(err) == 0
        compare(bf16_tensor_to_f64(out), _oracle_rows(b), what=f"call {i}: h={hist} q={q}")


@pytest.mark.parametrize("what", ["seq_lt_query", "seq_gt_table", "tokens"])
def test_validation_flags(cuda_lib, what):
    """Invalid lengths are flagged by the self-planning kernel and nothing is attended."""
    import torch
    spec = W.BatchSpec(hist=[100], qlen=[200], num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                       seed=1600)
    b = W.make_batch(spec)
    kc = to_dev(W.empty_cache(b).view(np.int16)).view(torch.bfloat16)
    vc = kc.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ql, sl = b.query_lens.copy(), b.seq_lens.copy()
    expect = {"seq_lt_query": cuda_lib.DEV_SEQ_LT_QUERY, "seq_gt_table": cuda_lib.DEV_SEQ_GT_TABLE,
              "tokens": cuda_lib.DEV_TOKENS_MISMATCH}[what]
    if what == "seq_lt_query":
        sl[0] = ql[0] - 1
    elif what == "seq_gt_table":
        sl[0] = b.block_table.shape[1] * 16 + 1
    else:
        ql[0] = 150          # num_tokens stays 200
    out = torch.zeros((200, 32, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(cuda_lib.cpp_attn_workspace_bytes(1, 200, 32, 8, 128, 8), dtype=torch.uint8, device="cuda")
    cuda_lib.cpp_chunked_prefill_attn(to_dev_bf16(b.q), kc, vc, to_dev(ql), to_dev(sl), to_dev(b.block_table), out,
                                      ws, err, max_kv_splits=8)
    torch.cuda.synchronize()
    assert cuda_lib.cpp_read_device_error(err) == expect
    assert bool((out == 0).all()), "an invalid request was attended"
