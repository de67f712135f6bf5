"""GPU parity of cpp_chunked_prefill_attn_write_kv, the KV write fused into the
attention call.

Two things are checked on every batch: the attention output against the fp64
oracle (the oracle's KV write of the new tokens, then its paged attention), and
the caches after the call against the oracle's KV write, bit for bit (slots
nobody writes keep their NaN pattern). The caches start as NaN patterns, so a
new key read from an unwritten slot instead of from k/v shows up as NaN."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import (cache_bits, compare, oracle_caches, run_gpu_batch, run_gpu_batch_fused, to_dev,
                     to_dev_bf16)

pytestmark = pytest.mark.gpu


def check_fused(cpsa, spec, max_kv_splits=8, scale=0.0):
    b = W.make_batch(spec)
    got, flags, kc, vc = run_gpu_batch_fused(cpsa, b, max_kv_splits=max_kv_splits, scale=scale)
    assert flags == 0, f"device flags {flags:#x}"
    okc, ovc = oracle_caches(b)
    assert np.array_equal(cache_bits(kc), okc) and np.array_equal(cache_bits(vc), ovc), "cache contents"
    ref = oracle.paged_attention(b.q, okc, ovc, b.query_lens, b.seq_lens, b.block_table, scale=scale)
    return compare(got, ref, what=spec.name or str(spec.qlen))


def test_fused_small_chunk(cuda_lib):
    check_fused(cuda_lib, W.spec_one_chunk_small())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (32, 8), (6, 2), (16, 1)])
def test_fused_heads_and_dims(cuda_lib, d, hq, hkv):
    """Histories off the 128 grid (130, 7) and on it (0); a decode row."""
    spec = W.BatchSpec(hist=[130, 0, 7], qlen=[200, 129, 1], num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                       page_size=16, seed=600 + hq + d)
    check_fused(cuda_lib, spec)


@pytest.mark.parametrize("P", [8, 16, 32, 64, 128, 256])
def test_fused_page_sizes(cuda_lib, P):
    spec = W.BatchSpec(hist=[300, 1000, 0], qlen=[77, 1, 260], num_q_heads=8, num_kv_heads=2, head_dim=128,
                       page_size=P, seed=700 + P, extra_pages=5)
    check_fused(cuda_lib, spec)


def test_fused_ragged_mixed_batch(cuda_lib):
    """Decode rows, chunks whose history ends inside a page and inside a 128-key tile,
    a zero-length request, a two-token prefill."""
    spec = W.BatchSpec(hist=[900, 33, 4000, 0, 511, 512, 513, 0, 77, 1],
                       qlen=[1, 1, 1, 2, 128, 127, 129, 0, 383, 2],
                       num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16, seed=800)
    check_fused(cuda_lib, spec)


@pytest.mark.parametrize("splits", [1, 2, 8])
def test_fused_long_history_splits(cuda_lib, splits):
    spec = W.BatchSpec(hist=[9000, 5000, 6001], qlen=[1, 150, 1], num_q_heads=8, num_kv_heads=2,
                       head_dim=128, page_size=16, seed=900 + splits)
    check_fused(cuda_lib, spec, max_kv_splits=splits)


def test_fused_decode_only(cuda_lib):
    rng = np.random.default_rng(13)
    ctx = [int(x) for x in rng.integers(1, 3000, size=40)]
    spec = W.BatchSpec(hist=[c - 1 for c in ctx], qlen=[1] * 40, num_q_heads=32, num_kv_heads=8, head_dim=128,
                       page_size=16, seed=901)
    check_fused(cuda_lib, spec)


def test_fused_tiny_prefills_and_scale(cuda_lib):
    spec = W.BatchSpec(hist=[0, 1, 2, 15, 16, 17], qlen=[2, 2, 3, 1, 5, 16], num_q_heads=4, num_kv_heads=1,
                       head_dim=64, page_size=8, seed=902)
    check_fused(cuda_lib, spec, scale=0.2)


def test_fused_matches_two_calls_bit_for_bit_on_the_128_grid(cuda_lib):
    """With every history a multiple of 128 the fused call tiles the keys as the
    two-call sequence does and reads the same bytes: identical outputs. Decode
    rows (any history) read the same bytes too."""
    import torch
    spec = W.BatchSpec(hist=[0, 128, 1024, 77, 3000], qlen=[300, 200, 129, 1, 1], num_q_heads=32,
                       num_kv_heads=8, head_dim=128, page_size=16, seed=903)
    b = W.make_batch(spec)
    a, fa, ka, va = run_gpu_batch(cuda_lib, b)
    f, ff, kf, vf = run_gpu_batch_fused(cuda_lib, b)
    assert fa == 0 and ff == 0
    assert np.array_equal(a.view(np.uint64), f.view(np.uint64))
    assert torch.equal(ka.view(torch.int16), kf.view(torch.int16))
    assert torch.equal(va.view(torch.int16), vf.view(torch.int16))


def test_fused_padding_and_out_of_range_slots(cuda_lib):
    """slot < 0 is skipped, a slot past the cache is flagged and skipped; the
    attention still uses those tokens' k/v (it reads the new rows directly)."""
    spec = W.BatchSpec(hist=[40, 300, 9], qlen=[150, 1, 70], num_q_heads=8, num_kv_heads=2, head_dim=64,
                       page_size=16, seed=904, extra_pages=2)
    b = W.make_batch(spec)
    slots = b.slot_mapping.copy()
    slots[3] = -1                    # a prefill token
    slots[140] = b.num_pages * 16    # a prefill token, past the cache
    slots[150] = -1                  # the decode row
    slots[160] = 10 ** 12
    got, flags, kc, vc = run_gpu_batch_fused(cuda_lib, b, slot_mapping=slots)
    assert flags == cuda_lib.DEV_SLOT_OUT_OF_RANGE
    okc, ovc = oracle_caches(b)
    ref = oracle.paged_attention(b.q, okc, ovc, b.query_lens, b.seq_lens, b.block_table)
    compare(got, ref, what="attention with skipped slots")
    ekc, evc = W.empty_cache(b), W.empty_cache(b)
    oracle.kv_cache_write(b.hist_k, b.hist_v, b.hist_slot_mapping, 16, ekc, evc)
    assert oracle.kv_cache_write(b.k, b.v, slots, 16, ekc, evc) == 2
    assert np.array_equal(cache_bits(kc), ekc) and np.array_equal(cache_bits(vc), evc)


def test_fused_null_inputs_rejected(cuda_lib):
    import torch
    lib = cuda_lib.load()
    p = lambda t: t.data_ptr()
    q = torch.zeros((4, 4, 64), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((2, 4, 16, 64), dtype=torch.bfloat16, device="cuda")
    ql = torch.tensor([4], dtype=torch.int32, device="cuda")
    bt = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    # k = NULL with tokens to write: rejected before any launch
    st = lib.cpp_chunked_prefill_attn_write_kv(p(q), None, p(q), p(ql), p(kc), p(kc), p(ql), p(ql), p(bt), 1, 4, 2,
                                               4, 4, 64, 16, 2, 0.0, 8, p(q), p(ws), ws.numel(), p(e), None)
    assert st == -1
    torch.cuda.synchronize()
    assert cuda_lib.cpp_read_device_error(e) == 0


def test_fused_llama_chunk_sampled_rows(cuda_lib):
    """Full size, the launch configuration the bench times: the 32768-token
    Llama-3-8B-shaped prompt (page 128) up to h = 8192 in fused 512-token steps;
    the last chunk's sampled rows against the oracle, and its cache rows bit for bit."""
    import torch
    SEQ, C, P, H = 32768, 512, 128, 8192
    q, k, v, slots, bt = W.device_sequence(SEQ, P)
    n_pages = bt.shape[1]
    kc = torch.full((n_pages, 8, P, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(cuda_lib.cpp_attn_workspace_bytes(1, C, 32, 8, 128, 8), dtype=torch.uint8, device="cuda")
    out = torch.empty((C, 32, 128), dtype=torch.bfloat16, device="cuda")
    ql = torch.tensor([C], dtype=torch.int32, device="cuda")
    for a in range(0, H + C, C):
        sl = torch.tensor([a + C], dtype=torch.int32, device="cuda")
        cuda_lib.cpp_chunked_prefill_attn_write_kv(q[a:a + C], k[a:a + C], v[a:a + C], slots[a:a + C], kc, vc, ql,
                                                   sl, bt, out, ws, err, max_kv_splits=8)
    torch.cuda.synchronize()
    assert cuda_lib.cpp_read_device_error(err) == 0
    u16 = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    # cache: the pages of the sequence so far hold k/v in token order
    s = H + C
    npg = s // P
    got_k = u16(kc[bt[0, :npg].long()])                              # [npg, 8, P, 128]
    want_k = u16(k[:s]).reshape(npg, P, 8, 128).transpose(0, 2, 1, 3)
    assert np.array_equal(got_k, want_k)
    got_v = u16(vc[bt[0, :npg].long()])
    want_v = u16(v[:s]).reshape(npg, P, 8, 128).transpose(0, 2, 1, 3)
    assert np.array_equal(got_v, want_v)
    rng = np.random.default_rng(77)
    rows = np.unique(np.concatenate([[0, 127, 128, 511], rng.choice(C, 12, replace=False)]))
    pos = np.arange(s)
    kk = np.full((npg, 8, P, 128), W.BF16_NAN_SENTINEL, dtype=np.uint16)
    vv = kk.copy()
    oracle.kv_cache_write(u16(k[:s]), u16(v[:s]), ((pos // P) * P + pos % P).astype(np.int64), P, kk, vv)
    ref = oracle.paged_attention(u16(q[H:s]), kk, vv, [C], [s], np.arange(npg, dtype=np.int32)[None, :],
                                 rows=rows)
    got = out[torch.from_numpy(rows).cuda()].float().cpu().numpy().astype(np.float64)
    compare(got, ref, what="fused llama chunk h=8192")


def test_fused_two_streams(cuda_lib):
    """AttentionStep with the fused call, two micro-batches on two streams, against one stream."""
    import torch
    spec = W.spec_microbatch()
    d = W.device_batch(spec)
    B, T = len(spec.qlen), sum(spec.qlen)
    kc0, vc0 = d["k_cache"].clone(), d["v_cache"].clone()
    step = cuda_lib.AttentionStep(B, T, 32, 8, 128, max_kv_splits=8, two_stream=True, fused_kv_write=True)
    out1 = torch.empty_like(d["q"])
    step.run(d["q"], d["k"], d["v"], d["slot_mapping"], d["k_cache"], d["v_cache"], d["query_lens"],
             d["seq_lens"], d["block_table"], out1)
    kc1, vc1 = d["k_cache"].clone(), d["v_cache"].clone()
    d["k_cache"].copy_(kc0)
    d["v_cache"].copy_(vc0)
    out2 = torch.empty_like(d["q"])
    used = step.run_two_stream(d["q"], d["k"], d["v"], d["slot_mapping"], d["k_cache"], d["v_cache"],
                               d["query_lens"], d["seq_lens"], d["block_table"], out2)
    torch.cuda.synchronize()
    assert used and step.read_errors() == 0
    assert torch.equal(kc1.view(torch.int16), d["k_cache"].view(torch.int16))
    assert torch.equal(vc1.view(torch.int16), d["v_cache"].view(torch.int16))
    compare(out2.float().cpu().numpy().astype(np.float64), out1.float().cpu().numpy().astype(np.float64),
            atol=1e-2, rtol_f=2e-3, what="fused: two streams vs one")
    # and the unfused step on the same input state agrees
    d["k_cache"].copy_(kc0)
    d["v_cache"].copy_(vc0)
    plain = cuda_lib.AttentionStep(B, T, 32, 8, 128, max_kv_splits=8)
    out3 = torch.empty_like(d["q"])
    plain.run(d["q"], d["k"], d["v"], d["slot_mapping"], d["k_cache"], d["v_cache"], d["query_lens"],
              d["seq_lens"], d["block_table"], out3)
    torch.cuda.synchronize()
    assert torch.equal(kc1.view(torch.int16), d["k_cache"].view(torch.int16))
    compare(out1.float().cpu().numpy().astype(np.float64), out3.float().cpu().numpy().astype(np.float64),
            atol=1e-2, rtol_f=2e-3, what="fused vs two calls")


def test_fused_events_entry_point(cuda_lib):
    """cpp_chunked_prefill_attn_write_kv_events (plain stream order) gives the same bits."""
    import torch
    spec = W.BatchSpec(hist=[900, 130, 0], qlen=[1, 300, 2], num_q_heads=8, num_kv_heads=2, head_dim=128,
                       page_size=16, seed=905)
    b = W.make_batch(spec)
    a, fa, ka, va = run_gpu_batch_fused(cuda_lib, b)
    kc = to_dev(W.empty_cache(b).view(np.int16)).view(torch.bfloat16)
    vc = kc.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cuda_lib.cpp_kv_cache_write(to_dev_bf16(b.hist_k), to_dev_bf16(b.hist_v), to_dev(b.hist_slot_mapping), kc, vc,
                                err)
    ws = torch.empty(cuda_lib.cpp_attn_workspace_bytes(3, b.num_tokens, 8, 2, 128, 8), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty((b.num_tokens, 8, 128), dtype=torch.bfloat16, device="cuda")
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    cuda_lib.cpp_chunked_prefill_attn_write_kv(to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v),
                                               to_dev(b.slot_mapping), kc, vc, to_dev(b.query_lens),
                                               to_dev(b.seq_lens), to_dev(b.block_table), out, ws, err,
                                               events=evs)
    torch.cuda.synchronize()
    assert fa == 0 and cuda_lib.cpp_read_device_error(err) == 0
    assert evs[1].elapsed_time(evs[2]) > 0
    assert np.array_equal(a.view(np.uint64), out.float().cpu().numpy().astype(np.float64).view(np.uint64))
    assert torch.equal(ka.view(torch.int16), kc.view(torch.int16))
    assert torch.equal(va.view(torch.int16), vc.view(torch.int16))


def test_fused_workspace_clamp(cuda_lib):
    """A workspace with room for the work lists only: nothing is split (flagged),
    the output and the caches are still right."""
    spec = W.BatchSpec(hist=[9000, 5000, 70], qlen=[1, 150, 300], num_q_heads=8, num_kv_heads=2, head_dim=128,
                       page_size=16, seed=906)
    b = W.make_batch(spec)
    minb = cuda_lib.cpp_attn_workspace_min_bytes(3, b.num_tokens, 8, 2, 128, 8)
    got, flags, kc, vc = run_gpu_batch_fused(cuda_lib, b, workspace_bytes=minb)
    assert flags == cuda_lib.DEV_SPLITS_CLAMPED
    okc, ovc = oracle_caches(b)
    assert np.array_equal(cache_bits(kc), okc) and np.array_equal(cache_bits(vc), ovc)
    ref = oracle.paged_attention(b.q, okc, ovc, b.query_lens, b.seq_lens, b.block_table)
    compare(got, ref, what="fused, clamped workspace")
