"""The batch builder feeding the kernels step after step (closed loop): every step's
metadata comes from the library's scheduler, the step's new K/V go through
cpp_kv_cache_write and its rows through cpp_chunked_prefill_attn (or both
through the fused cpp_chunked_prefill_attn_write_kv); the oracle replays the
same writes into its own cache and checks every output row of every step, and
the caches bit for bit at the end. Covers decode rows mixed with prompts that span several steps, pages
allocated as sequences grow and reused after requests finish."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import bf16_tensor_to_f64, compare, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

HQ, HKV, D, P = 8, 2, 64, 16


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("budget,caps,tile", [(256, (), 0), (512, (256, 128, 64), 16)])
def test_scheduler_feeds_the_kernels(cuda_lib, budget, caps, tile, fused):
    import torch
    pages = 160                      # small pool: pages must be reused after requests finish
    rng = np.random.Generator(np.random.PCG64(77 + budget))
    order = rng.permutation(pages).astype(np.int32)
    sched = cuda_lib.BatchScheduler(budget, P, pages, page_order=order, chunk_caps=caps, tile_align=tile,
                                    max_reqs=64, max_blocks=128)
    prompts = [(0, 300, 3), (1, 57, 5), (2, 700, 0), (3, 129, 2), (4, 1, 4), (5, 450, 1), (6, 900, 2), (7, 33, 6)]
    for rid, L, m in prompts:
        sched.add_request(rid, L, m)
    # both sides start from the same NaN pattern, so unwritten slots compare equal too
    okc = np.full((pages, HKV, P, D), W.BF16_NAN_SENTINEL, dtype=np.uint16)
    okv = okc.copy()
    kc = to_dev(okc.view(np.int16)).view(torch.bfloat16)
    vc = kc.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    steps, decode_rows = 0, 0
    while True:
        waiting, running, finished, free = sched.stats()
        if waiting == 0 and running == 0:
            break
        b = sched.step()
        B, T = len(b["req_ids"]), len(b["slot_mapping"])
        assert B > 0, "no progress"
        q = W.randn_bf16(rng, (T, HQ, D))
        k = W.randn_bf16(rng, (T, HKV, D))
        v = W.randn_bf16(rng, (T, HKV, D))
        ws = torch.empty(cuda_lib.cpp_attn_workspace_bytes(B, T, HQ, HKV, D, 8), dtype=torch.uint8, device="cuda")
        out = torch.full((T, HQ, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        if fused:
            cuda_lib.cpp_chunked_prefill_attn_write_kv(to_dev_bf16(q), to_dev_bf16(k), to_dev_bf16(v),
                                                       to_dev(b["slot_mapping"]), kc, vc, to_dev(b["query_lens"]),
                                                       to_dev(b["seq_lens"]), to_dev(b["block_table"]), out, ws, err,
                                                       max_kv_splits=8)
        else:
            cuda_lib.cpp_kv_cache_write(to_dev_bf16(k), to_dev_bf16(v), to_dev(b["slot_mapping"]), kc, vc, err)
            cuda_lib.cpp_chunked_prefill_attn(to_dev_bf16(q), kc, vc, to_dev(b["query_lens"]), to_dev(b["seq_lens"]),
                                              to_dev(b["block_table"]), out, ws, err, max_kv_splits=8)
        oracle.kv_cache_write(k, v, b["slot_mapping"], P, okc, okv)
        ref = oracle.paged_attention(q, okc, okv, b["query_lens"], b["seq_lens"], b["block_table"])
        torch.cuda.synchronize()
        compare(bf16_tensor_to_f64(out), ref, what=f"step {steps}")
        decode_rows += int((b["query_lens"] == 1).sum())
        sched.commit()
        steps += 1
        assert steps < 200
    assert cuda_lib.cpp_read_device_error(err) == 0
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(bits(kc), okc) and np.array_equal(bits(vc), okv), "caches after the loop"
    assert sched.stats() == (0, 0, len(prompts), pages)
    assert decode_rows >= sum(m for _, _, m in prompts)
    sched.close()
