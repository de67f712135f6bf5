"""GPU parity at the full workload sizes, in the launch configuration bench.py
times, on sampled rows that the fp64 oracle computes one by one.

For every sampled request the oracle gets that request's own inputs: its
history K/V (read from the cache pages BEFORE this step's KV write, i.e. the
seeded input state) and its new tokens' q/k/v; it writes the new tokens with
its own KV write into a compact cache and evaluates the sampled rows."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import compare

pytestmark = pytest.mark.gpu


def _u16(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_rows(q_req, k_new, v_new, hist_pages_k, hist_pages_v, hist, qlen, P, rows):
    """Oracle attention of rows `rows` (0-based within the request) of one request.

    hist_pages_*: uint16 [n_pages, Hkv, P, d] -- the request's pages in block
    order, holding its history; new tokens go to positions hist .. hist+qlen-1."""
    n_pages = hist_pages_k.shape[0]
    kc = hist_pages_k.copy()
    vc = hist_pages_v.copy()
    pos = np.arange(hist, hist + qlen)
    slots = (pos // P) * P + pos % P                      # identity page table 0..n-1
    assert oracle.kv_cache_write(k_new, v_new, slots.astype(np.int64), P, kc, vc) == 0
    bt = np.arange(n_pages, dtype=np.int32)[None, :]
    return oracle.paged_attention(q_req, kc, vc, [qlen], [hist + qlen], bt, rows=np.asarray(rows))


@pytest.mark.parametrize("history", [0, 512, 8192, 32256])
def test_llama_chunk_sampled_rows(cuda_lib, history):
    """One 512-token chunk of the 32768-token Llama-3-8B-shaped prefill (page 128)."""
    import torch
    SEQ, C, P = 32768, 512, 128
    q, k, v, slots, bt = W.device_sequence(SEQ, P)
    n_pages = bt.shape[1]
    kc = torch.full((n_pages, 8, P, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # history written chunk by chunk, exactly as the step does
    for a in range(0, history + C, C):
        cuda_lib.cpp_kv_cache_write(k[a:a + C], v[a:a + C], slots[a:a + C], kc, vc, err)
    out = torch.empty((C, 32, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(cuda_lib.cpp_attn_workspace_bytes(1, C, 32, 8, 128, 8), dtype=torch.uint8, device="cuda")
    ql = torch.tensor([C], dtype=torch.int32, device="cuda")
    sl = torch.tensor([history + C], dtype=torch.int32, device="cuda")
    cuda_lib.cpp_chunked_prefill_attn(q[history:history + C], kc, vc, ql, sl, bt, out, ws, err, max_kv_splits=8)
    torch.cuda.synchronize()
    assert cuda_lib.cpp_read_device_error(err) == 0
    rng = np.random.default_rng(history)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, 383, 384, 510, 511],
                                     rng.choice(C, 22, replace=False)]))
    # oracle: the sequence prefix in token order (its own KV write, identity pages)
    s = history + C
    npg = (s + P - 1) // P
    kk = np.full((npg, 8, P, 128), W.BF16_NAN_SENTINEL, dtype=np.uint16)
    vv = kk.copy()
    if history:
        pos = np.arange(0, history)
        oracle.kv_cache_write(_u16(k[:history]), _u16(v[:history]), ((pos // P) * P + pos % P).astype(np.int64),
                              P, kk, vv)
    ref = oracle_rows(_u16(q[history:s]), _u16(k[history:s]), _u16(v[history:s]), kk, vv, history, C, P, rows)
    got = out[torch.from_numpy(rows).cuda()].float().cpu().numpy().astype(np.float64)
    compare(got, ref, what=f"llama chunk h={history}")


def _sampled_parity(cuda_lib, spec, sample_reqs, rows_per_req, seed, fused=False):
    import torch
    d = W.device_batch(spec)
    B, T = len(spec.qlen), sum(spec.qlen)
    P = spec.page_size
    bt = d["block_table_host"]
    # input state of the sampled requests' pages, before this step's KV write
    saved = {}
    for r in sample_reqs:
        npg = (spec.seq[r] + P - 1) // P
        idx = torch.from_numpy(bt[r, :npg].astype(np.int64)).cuda()
        saved[r] = (_u16(d["k_cache"][idx]), _u16(d["v_cache"][idx]))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(d["q"])
    ws = torch.empty(cuda_lib.cpp_attn_workspace_bytes(B, T, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, 8),
                     dtype=torch.uint8, device="cuda")
    if fused:
        cuda_lib.cpp_chunked_prefill_attn_write_kv(d["q"], d["k"], d["v"], d["slot_mapping"], d["k_cache"],
                                                   d["v_cache"], d["query_lens"], d["seq_lens"], d["block_table"],
                                                   out, ws, err, max_kv_splits=8)
    else:
        cuda_lib.cpp_kv_cache_write(d["k"], d["v"], d["slot_mapping"], d["k_cache"], d["v_cache"], err)
        cuda_lib.cpp_chunked_prefill_attn(d["q"], d["k_cache"], d["v_cache"], d["query_lens"], d["seq_lens"],
                                          d["block_table"], out, ws, err, max_kv_splits=8)
    torch.cuda.synchronize()
    assert cuda_lib.cpp_read_device_error(err) == 0
    # the sampled requests' new rows sit in their cache slots, bit for bit
    cu0 = np.concatenate([[0], np.cumsum(spec.qlen)])
    slots_h = d["slot_mapping"].cpu().numpy()
    for r in sample_reqs:
        t0, t1 = int(cu0[r]), int(cu0[r + 1])
        s = torch.from_numpy(slots_h[t0:t1]).cuda()
        rows_k = d["k_cache"][s // P, :, s % P]          # [tokens, Hkv, D]
        rows_v = d["v_cache"][s // P, :, s % P]
        assert torch.equal(rows_k.view(torch.int16), d["k"][t0:t1].view(torch.int16))
        assert torch.equal(rows_v.view(torch.int16), d["v"][t0:t1].view(torch.int16))
    cu = np.concatenate([[0], np.cumsum(spec.qlen)])
    rng = np.random.default_rng(seed)
    gots, refs = [], []
    for r in sample_reqs:
        ql, h = spec.qlen[r], spec.hist[r]
        rows = np.arange(ql) if ql <= rows_per_req else np.unique(
            np.concatenate([[0, ql - 1], rng.choice(ql, rows_per_req, replace=False)]))
        t0, t1 = int(cu[r]), int(cu[r + 1])
        hk, hv = saved[r]
        ref = oracle_rows(_u16(d["q"][t0:t1]), _u16(d["k"][t0:t1]), _u16(d["v"][t0:t1]), hk, hv, h, ql, P, rows)
        got = out[t0 + torch.from_numpy(rows).cuda()].float().cpu().numpy().astype(np.float64)
        gots.append(got)
        refs.append(ref)
    return np.concatenate(gots), np.concatenate(refs), d, out


@pytest.mark.parametrize("fused", [False, True])
def test_sarathi_mixed_sampled(cuda_lib, fused):
    """1536 decode rows (context U[1024, 8192]) + one 512-token chunk at h = 8192, page 16;
    the KV write as its own call or fused into the attention call."""
    spec = W.spec_sarathi_mixed()
    rng = np.random.default_rng(33)
    reqs = sorted(set(rng.choice(1536, 24, replace=False).tolist()) | {0, 1535, 1536})
    got, ref, _, _ = _sampled_parity(cuda_lib, spec, reqs, rows_per_req=24, seed=34, fused=fused)
    compare(got, ref, what="sarathi mixed" + (" (fused)" if fused else ""))


@pytest.mark.parametrize("fused", [False, True])
def test_microbatch_sampled(cuda_lib, fused):
    """128 decode rows (context U[2600, 5200]) + 64 prompts of 2600 tokens, page 16."""
    spec = W.spec_microbatch()
    reqs = [0, 5, 77, 127, 128, 150, 191]
    got, ref, _, _ = _sampled_parity(cuda_lib, spec, reqs, rows_per_req=16, seed=35, fused=fused)
    compare(got, ref, what="microbatch" + (" (fused)" if fused else ""))


def _saved_pages(spec, d, reqs):
    """The sampled requests' cache pages as they are before this step's KV write
    (the seeded input state the oracle starts from)."""
    import torch
    P = spec.page_size
    bt = d["block_table_host"]
    saved = {}
    for r in reqs:
        npg = (spec.seq[r] + P - 1) // P
        idx = torch.from_numpy(bt[r, :npg].astype(np.int64)).cuda()
        saved[r] = (_u16(d["k_cache"][idx]), _u16(d["v_cache"][idx]))
    return saved


def _oracle_picks(spec, d, out, saved, picks):
    """(got, ref) of the rows picks[r] (0-based within request r) of `out`."""
    import torch
    cu = np.concatenate([[0], np.cumsum(spec.qlen)])
    gots, refs = [], []
    for r, rows in picks.items():
        ql, h = spec.qlen[r], spec.hist[r]
        t0, t1 = int(cu[r]), int(cu[r + 1])
        hk, hv = saved[r]
        ref = oracle_rows(_u16(d["q"][t0:t1]), _u16(d["k"][t0:t1]), _u16(d["v"][t0:t1]), hk, hv, h, ql,
                          spec.page_size, rows)
        got = out[t0 + torch.from_numpy(np.asarray(rows)).cuda()].float().cpu().numpy().astype(np.float64)
        gots.append(got)
        refs.append(ref)
    return np.concatenate(gots), np.concatenate(refs)


@pytest.mark.parametrize("fused", [False, True])
def test_two_streams_match_oracle(cuda_lib, fused):
    """The micro-batch workload (128 decode rows, then 64 prompts of 2600) split at
    the balanced point (160, 83328) and run as two micro-batches on two streams
    ("Ascend dual-stream parallel" article, section 3.1: requests before the
    split and tokens before token_split form micro-batch 0), with the KV write as
    its own call or fused: sampled rows against the fp64 oracle -- the decode
    rows of 8 decode requests and 16 rows (0 and 2599 among them) of 6 prompts,
    three in each micro-batch -- and against the one-stream run.

    The prefill work is cut into equal runs per CTA over each call's batch, so
    the two micro-batches cut their units elsewhere than the full batch does:
    two-stream and one-stream outputs agree within the attention tolerance, and
    decode rows (split by their own length only) bit for bit."""
    import torch
    spec = W.spec_microbatch()
    d = W.device_batch(spec)
    B, T = len(spec.qlen), sum(spec.qlen)
    dec_reqs = [0, 9, 31, 58, 64, 100, 126, 127]
    pre_reqs = [128, 141, 159, 160, 177, 191]        # 128..159: micro-batch 0; 160..191: micro-batch 1
    saved = _saved_pages(spec, d, dec_reqs + pre_reqs)
    step = cuda_lib.AttentionStep(B, T, 32, 8, 128, max_kv_splits=8, two_stream=True, fused_kv_write=fused)
    # the first KV write happens in both runs (the same bytes); history pages are read-only
    out1 = torch.empty_like(d["q"])
    step.run(d["q"], d["k"], d["v"], d["slot_mapping"], d["k_cache"], d["v_cache"], d["query_lens"],
             d["seq_lens"], d["block_table"], out1)
    out2 = torch.full_like(d["q"], float("nan"))
    used = step.run_two_stream(d["q"], d["k"], d["v"], d["slot_mapping"], d["k_cache"], d["v_cache"],
                               d["query_lens"], d["seq_lens"], d["block_table"], out2)
    torch.cuda.synchronize()
    assert used and step.last_split == (160, 83328, True)
    assert step.read_errors() == 0
    rng = np.random.default_rng(36 + int(fused))
    picks = {r: [0] for r in dec_reqs}
    for r in pre_reqs:
        ql = spec.qlen[r]
        picks[r] = np.unique(np.concatenate([[0, ql - 1], rng.choice(np.arange(1, ql - 1), 14, replace=False)]))
        assert len(picks[r]) == 16
    got, ref = _oracle_picks(spec, d, out2, saved, picks)
    compare(got, ref, what="two streams vs oracle" + (" (fused)" if fused else ""))
    got1, _ = _oracle_picks(spec, d, out1, saved, picks)
    compare(got1, ref, what="one stream vs oracle" + (" (fused)" if fused else ""))
    compare(out2.float().cpu().numpy().astype(np.float64), out1.float().cpu().numpy().astype(np.float64),
            atol=1e-2, rtol_f=2e-3, what="two streams vs one")
    n_dec = 128
    assert torch.equal(out1[:n_dec].view(torch.int16), out2[:n_dec].view(torch.int16))
    # the same run with the split passed in (computed once per batch): identical bits
    out3 = torch.full_like(d["q"], float("nan"))
    assert step.run_two_stream(d["q"], d["k"], d["v"], d["slot_mapping"], d["k_cache"], d["v_cache"],
                               d["query_lens"], d["seq_lens"], d["block_table"], out3, split=step.last_split)
    torch.cuda.synchronize()
    assert step.read_errors() == 0
    assert torch.equal(out3.view(torch.int16), out2.view(torch.int16))


def test_gpu_chunk_invariance(cuda_lib):
    """A 2048-token prompt prefilled as one chunk or as four chunks of 512 agrees."""
    import torch
    q, k, v, slots, bt = W.device_sequence(2048, 16, seed=9)
    n_pages = bt.shape[1]
    outs = []
    for chunk in (2048, 512):
        kc = torch.full((n_pages, 8, 16, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        vc = kc.clone()
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.empty_like(q)
        ws = torch.empty(cuda_lib.cpp_attn_workspace_bytes(1, chunk, 32, 8, 128, 8), dtype=torch.uint8,
                         device="cuda")
        for a in range(0, 2048, chunk):
            cuda_lib.cpp_kv_cache_write(k[a:a + chunk], v[a:a + chunk], slots[a:a + chunk], kc, vc, err)
            cuda_lib.cpp_chunked_prefill_attn(q[a:a + chunk], kc, vc, torch.tensor([chunk], dtype=torch.int32,
                                                                                    device="cuda"),
                                              torch.tensor([a + chunk], dtype=torch.int32, device="cuda"), bt,
                                              out[a:a + chunk], ws, err)
        torch.cuda.synchronize()
        assert cuda_lib.cpp_read_device_error(err) == 0
        outs.append(out.float().cpu().numpy().astype(np.float64))
    compare(outs[1], outs[0], atol=1e-2, rtol_f=3e-3, what="chunked vs whole")


def test_llama_64_chunks_match_one_prefill(cuda_lib):
    """The headline workload end to end: the 32768-token prompt prefilled in 64
    fused chunks of 512 agrees with the same prompt prefilled as one causal chunk
    of 32768 (every row, every head), and both leave the same cache."""
    import torch
    SEQ, C, P = 32768, 512, 128
    q, k, v, slots, bt = W.device_sequence(SEQ, P)
    n_pages = bt.shape[1]
    outs, caches = [], []
    for chunk in (C, SEQ):
        kc = torch.full((n_pages, 8, P, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        vc = kc.clone()
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.empty_like(q)
        ws = torch.empty(cuda_lib.cpp_attn_workspace_bytes(1, chunk, 32, 8, 128, 8), dtype=torch.uint8,
                         device="cuda")
        ql = torch.tensor([chunk], dtype=torch.int32, device="cuda")
        for a in range(0, SEQ, chunk):
            sl = torch.tensor([a + chunk], dtype=torch.int32, device="cuda")
            cuda_lib.cpp_chunked_prefill_attn_write_kv(q[a:a + chunk], k[a:a + chunk], v[a:a + chunk],
                                                       slots[a:a + chunk], kc, vc, ql, sl, bt, out[a:a + chunk],
                                                       ws, err, max_kv_splits=8)
        torch.cuda.synchronize()
        assert cuda_lib.cpp_read_device_error(err) == 0
        outs.append(out)
        caches.append((kc, vc))
    assert torch.equal(caches[0][0].view(torch.int16), caches[1][0].view(torch.int16))
    assert torch.equal(caches[0][1].view(torch.int16), caches[1][1].view(torch.int16))
    a, b = outs[0].float(), outs[1].float()
    assert bool(torch.isfinite(a).all()) and bool(torch.isfinite(b).all())
    max_abs = float((a - b).abs().max())
    rel_f = float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(b))
    assert max_abs <= 1e-2 and rel_f <= 3e-3, f"64 chunks vs one: max-abs {max_abs:.3e} rel-F {rel_f:.3e}"


def test_dynamic_chunks_sampled_rows(cuda_lib):
    """The dynamic-chunking workload: the 32768-token prompt (page 128) in the
    chunk sizes the planner gives for a fixed quadratic latency model, fused
    calls; sampled rows of every chunk (first, last and six drawn) against the
    oracle."""
    import torch
    SEQ, P = 32768, 128
    # a latency model of the size the profile fits give on this GPU (ms)
    chunks = cuda_lib.cpp_plan_chunk_sizes(4.75e-9, 3.87e-5, 0.024, SEQ, 4096, P, 64, 0, 0, 1.0)
    assert sum(chunks) == SEQ and chunks[0] == 4096 and len(chunks) > 8
    q, k, v, slots, bt = W.device_sequence(SEQ, P, seed=4)
    n_pages = bt.shape[1]
    kc = torch.full((n_pages, 8, P, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    ws = torch.empty(cuda_lib.cpp_attn_workspace_bytes(1, max(chunks), 32, 8, 128, 8), dtype=torch.uint8,
                     device="cuda")
    a = 0
    for c in chunks:
        ql = torch.tensor([c], dtype=torch.int32, device="cuda")
        sl = torch.tensor([a + c], dtype=torch.int32, device="cuda")
        cuda_lib.cpp_chunked_prefill_attn_write_kv(q[a:a + c], k[a:a + c], v[a:a + c], slots[a:a + c], kc, vc,
                                                   ql, sl, bt, out[a:a + c], ws, err, max_kv_splits=8)
        a += c
    torch.cuda.synchronize()
    assert cuda_lib.cpp_read_device_error(err) == 0
    rng = np.random.default_rng(44)
    rows = []
    a = 0
    for c in chunks:
        rows.extend([a, a + c - 1] + [a + int(x) for x in rng.choice(c, 6, replace=False)])
        a += c
    rows = np.unique(np.asarray(rows))
    n_pg = SEQ // P
    kk = np.full((n_pg, 8, P, 128), W.BF16_NAN_SENTINEL, dtype=np.uint16)
    vv = kk.copy()
    pos = np.arange(SEQ)
    oracle.kv_cache_write(_u16(k), _u16(v), ((pos // P) * P + pos % P).astype(np.int64), P, kk, vv)
    # the whole prompt as one request: row t sees keys 0..t, whichever chunk held it
    ref = oracle.paged_attention(_u16(q), kk, vv, [SEQ], [SEQ], np.arange(n_pg, dtype=np.int32)[None, :],
                                 rows=rows)
    got = out[torch.from_numpy(rows).cuda()].float().cpu().numpy().astype(np.float64)
    compare(got, ref, what="dynamic chunks")


def test_fused_headline_step_sampled_rows(cuda_lib):
    """The headline step exactly as the bench runs it (64 fused chunks of 512,
    page 128, max_kv_splits 8): 64 rows of chunks 0, 1, 7, 31 and 63 (rows 0,
    127, 128 and 511 always among them) against the oracle, and the cache bit for
    bit after the last chunk."""
    import torch
    SEQ, C, P = 32768, 512, 128
    q, k, v, slots, bt = W.device_sequence(SEQ, P)
    n_pages = bt.shape[1]
    kc = torch.full((n_pages, 8, P, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(cuda_lib.cpp_attn_workspace_bytes(1, C, 32, 8, 128, 8), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    ql = torch.tensor([C], dtype=torch.int32, device="cuda")
    for a in range(0, SEQ, C):
        sl = torch.tensor([a + C], dtype=torch.int32, device="cuda")
        cuda_lib.cpp_chunked_prefill_attn_write_kv(q[a:a + C], k[a:a + C], v[a:a + C], slots[a:a + C], kc, vc, ql,
                                                   sl, bt, out[a:a + C], ws, err, max_kv_splits=8)
    torch.cuda.synchronize()
    assert cuda_lib.cpp_read_device_error(err) == 0
    # cache: page bt[0, j] holds positions j*P .. j*P+P-1 of the prompt
    npg = SEQ // P
    assert np.array_equal(_u16(kc[bt[0].long()]), _u16(k).reshape(npg, P, 8, 128).transpose(0, 2, 1, 3))
    assert np.array_equal(_u16(vc[bt[0].long()]), _u16(v).reshape(npg, P, 8, 128).transpose(0, 2, 1, 3))
    # oracle: the whole prompt as one request on identity pages; row t sees keys 0..t
    kk = np.full((npg, 8, P, 128), W.BF16_NAN_SENTINEL, dtype=np.uint16)
    vv = kk.copy()
    pos = np.arange(SEQ)
    oracle.kv_cache_write(_u16(k), _u16(v), ((pos // P) * P + pos % P).astype(np.int64), P, kk, vv)
    rng = np.random.default_rng(63)
    rows = []
    for ci in (0, 1, 7, 31, 63):
        fixed = np.array([0, 127, 128, C - 1])
        pick = np.concatenate([fixed, rng.choice(np.setdiff1d(np.arange(C), fixed), 60, replace=False)])
        rows.append(ci * C + pick)
    rows = np.sort(np.concatenate(rows))
    ref = oracle.paged_attention(_u16(q), kk, vv, [SEQ], [SEQ], np.arange(npg, dtype=np.int32)[None, :], rows=rows)
    got = out[torch.from_numpy(rows).cuda()].float().cpu().numpy().astype(np.float64)
    compare(got, ref, what="headline step, sampled rows")
