"""Pins of the fp64 oracle's KV write and attention to facts fixed outside it.

Every test here runs on the CPU. Each case is chosen so that a plausible slip in
the oracle fails at least one of them:
  scale (1/sqrt(d))            -> hand 2x2 example
  causal offset / off-by-one   -> hand 2x2 example, chunk invariance, history case
  page gather (page vs offset) -> hand example (block_table [1, 0]), page relabelling
  GQA head mapping             -> per-kv-head constant values; GQA = MHA with repeated kv heads
  softmax normalisation        -> one-hot values (probabilities sum to 1), constant V
  max subtraction / overflow   -> huge scores reduce to the argmax key's value
  KV write layout              -> hand-placed slots, sentinel bytes untouched
"""
import math
import os

import numpy as np
import pytest

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf(x):
    return W.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def build_cache_and_run(batch, rows=None, scale=0.0):
    kc = W.empty_cache(batch)
    vc = W.empty_cache(batch)
    P = batch.spec.page_size
    if batch.hist_k is not None and batch.hist_k.shape[0]:
        assert oracle.kv_cache_write(batch.hist_k, batch.hist_v, batch.hist_slot_mapping, P, kc, vc) == 0
    assert oracle.kv_cache_write(batch.k, batch.v, batch.slot_mapping, P, kc, vc) == 0
    out = oracle.paged_attention(batch.q, kc, vc, batch.query_lens, batch.seq_lens,
                                 batch.block_table, scale=scale, rows=rows)
    return out, kc, vc


def load_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(x) for x in line.split()])
    return np.asarray(rows)


def test_hand_2x2_example():
    q = bf([[[1.0, 0.0]], [[0.0, 1.0]]])           # [T=2, Hq=1, d=2]
    k = bf([[[1.0, 0.0]], [[0.0, 1.0]]])
    v = bf([[[1.0, 2.0]], [[3.0, 4.0]]])
    bt = np.array([[1, 0]], dtype=np.int32)
    slots = np.array([1, 0], dtype=np.int64)        # token 0 -> page 1, token 1 -> page 0
    kc = np.full((2, 1, 1, 2), W.BF16_NAN_SENTINEL, dtype=np.uint16)
    vc = kc.copy()
    assert oracle.kv_cache_write(k, v, slots, 1, kc, vc) == 0
    out = oracle.paged_attention(q, kc, vc, [2], [2], bt)
    gold = load_golden("hand_2x2.txt")
    np.testing.assert_allclose(out[:, 0, :], gold[:, 1:], rtol=0, atol=1e-14)


def test_hand_example_with_history():
    # the same token 1 asked as a one-token chunk after a one-token history
    q = bf([[[0.0, 1.0]]])
    hk = bf([[[1.0, 0.0]]]); hv = bf([[[1.0, 2.0]]])
    k = bf([[[0.0, 1.0]]]); v = bf([[[3.0, 4.0]]])
    kc = np.full((2, 1, 1, 2), W.BF16_NAN_SENTINEL, dtype=np.uint16)
    vc = kc.copy()
    oracle.kv_cache_write(hk, hv, np.array([1]), 1, kc, vc)
    oracle.kv_cache_write(k, v, np.array([0]), 1, kc, vc)
    out = oracle.paged_attention(q, kc, vc, [1], [2], np.array([[1, 0]], dtype=np.int32))
    gold = load_golden("hand_2x2.txt")
    np.testing.assert_allclose(out[0, 0], gold[1, 1:], rtol=0, atol=1e-14)


def test_single_key_returns_value_exactly():
    rng = np.random.default_rng(0)
    q = W.randn_bf16(rng, (1, 2, 8)); k = W.randn_bf16(rng, (1, 1, 8)); v = W.randn_bf16(rng, (1, 1, 8))
    kc = np.full((1, 1, 4, 8), W.BF16_NAN_SENTINEL, dtype=np.uint16); vc = kc.copy()
    oracle.kv_cache_write(k, v, np.array([0]), 4, kc, vc)
    out = oracle.paged_attention(q, kc, vc, [1], [1], np.array([[0]], dtype=np.int32))
    want = W.bf16_bits_to_f32(v[0, 0]).astype(np.float64)
    assert np.array_equal(out[0, 0], want) and np.array_equal(out[0, 1], want)


def test_constant_values_return_the_constant():
    spec = W.BatchSpec(hist=[37, 0], qlen=[20, 33], num_q_heads=4, num_kv_heads=2, head_dim=16,
                       page_size=8, seed=11)
    b = W.make_batch(spec)
    const = bf(np.linspace(-3, 3, 16))
    b.v[:] = const; b.hist_v[:] = const
    out, _, _ = build_cache_and_run(b)
    np.testing.assert_allclose(out, np.broadcast_to(W.bf16_bits_to_f32(const), out.shape),
                               rtol=0, atol=1e-13)


def test_gqa_head_mapping_by_group():
    # kv head j carries the constant value j+1 -> q head h must return h // g + 1
    spec = W.BatchSpec(hist=[5], qlen=[7], num_q_heads=8, num_kv_heads=2, head_dim=4,
                       page_size=4, seed=12)
    b = W.make_batch(spec)
    for j in range(2):
        b.v[:, j, :] = bf(np.full(4, j + 1.0)); b.hist_v[:, j, :] = bf(np.full(4, j + 1.0))
    out, _, _ = build_cache_and_run(b)
    for h in range(8):
        assert np.allclose(out[:, h, :], h // 4 + 1.0, atol=1e-13, rtol=0)


def test_gqa_equals_mha_with_each_kv_head_repeated_for_its_group():
    # grouped-query attention is multi-head attention whose kv head h is the
    # grouped kv head h // g: the same rows, bit for bit, with every q head
    # scoring its own query row (random K/V, so no head is interchangeable)
    spec = W.BatchSpec(hist=[5, 0, 9], qlen=[7, 3, 1], num_q_heads=6, num_kv_heads=2, head_dim=8,
                       page_size=4, seed=17)
    b = W.make_batch(spec)
    out_gqa, kc, vc = build_cache_and_run(b)
    kc_mha = np.ascontiguousarray(np.repeat(kc, 3, axis=1))
    vc_mha = np.ascontiguousarray(np.repeat(vc, 3, axis=1))
    out_mha = oracle.paged_attention(b.q, kc_mha, vc_mha, b.query_lens, b.seq_lens, b.block_table)
    assert np.array_equal(out_gqa, out_mha)
    # and the heads of one group do differ (each reads its own query row)
    assert not np.allclose(out_gqa[:, 0, :], out_gqa[:, 1, :])


def test_one_hot_values_give_probabilities_that_sum_to_one():
    # d >= number of keys: value j = e_j, so the output row is the probability vector
    d = 32
    spec = W.BatchSpec(hist=[9], qlen=[12], num_q_heads=1, num_kv_heads=1, head_dim=d,
                       page_size=4, seed=13)
    b = W.make_batch(spec)
    eye = bf(np.eye(d))
    b.hist_v[:, 0, :] = eye[:9]
    b.v[:, 0, :] = eye[9:21]
    out, _, _ = build_cache_and_run(b)
    p = out[:, 0, :]
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    for i in range(12):
        assert np.all(p[i, : 9 + i + 1] > 0.0)          # every visible key has weight
        assert np.all(p[i, 9 + i + 1:] == 0.0)          # no future key has weight


def test_huge_scores_select_the_argmax_key():
    # scores of size ~1e4 overflow exp() unless the maximum is subtracted first
    d = 4
    q = bf([[[100.0, 0, 0, 0]]])
    hk = bf([[[1.0, 0, 0, 0]], [[100.0, 0, 0, 0]], [[-100.0, 0, 0, 0]]])
    hv = bf([[[1.0, 1, 1, 1]], [[7.0, 7, 7, 7]], [[-5.0, -5, -5, -5]]])
    k = bf([[[50.0, 0, 0, 0]]]); v = bf([[[2.0, 2, 2, 2]]])
    kc = np.full((1, 1, 4, d), W.BF16_NAN_SENTINEL, dtype=np.uint16); vc = kc.copy()
    oracle.kv_cache_write(hk, hv, np.array([0, 1, 2]), 4, kc, vc)
    oracle.kv_cache_write(k, v, np.array([3]), 4, kc, vc)
    out = oracle.paged_attention(q, kc, vc, [1], [4], np.array([[0]], dtype=np.int32))
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out[0, 0], 7.0, rtol=0, atol=1e-12)


def test_chunk_invariance_small_workload():
    """History 256 + chunk 128 equals the last 128 rows of one 384-token prefill."""
    spec = W.spec_one_chunk_small()
    chunked = W.make_batch(spec)
    out_c, _, _ = build_cache_and_run(chunked)
    # the same 384 tokens as one fresh prompt (same pages, same values)
    T = 384
    q_all = np.concatenate([W.randn_bf16(np.random.default_rng(99), (256, 4, 64)), chunked.q])
    whole = W.Batch(spec=W.BatchSpec(hist=[0], qlen=[T], num_q_heads=4, num_kv_heads=4,
                                     head_dim=64, page_size=16, seed=0),
                    q=q_all,
                    k=np.concatenate([chunked.hist_k, chunked.k]),
                    v=np.concatenate([chunked.hist_v, chunked.v]),
                    slot_mapping=np.concatenate([chunked.hist_slot_mapping, chunked.slot_mapping]),
                    block_table=chunked.block_table, query_lens=np.array([T], dtype=np.int32),
                    seq_lens=np.array([T], dtype=np.int32), num_pages=chunked.num_pages)
    out_w, _, _ = build_cache_and_run(whole, rows=np.arange(256, 384))
    assert np.array_equal(out_c, out_w)


def test_chunk_invariance_two_chunks_multi_request():
    spec = W.BatchSpec(hist=[0, 13], qlen=[40, 30], num_q_heads=4, num_kv_heads=2, head_dim=16,
                       page_size=8, seed=21)
    b = W.make_batch(spec)
    out_all, kc, vc = build_cache_and_run(b)
    # request 0 split as 25 + 15: ask the second piece with history 25
    rows0 = oracle.paged_attention(b.q[25:40], kc, vc, [15], [40], b.block_table[:1])
    assert np.array_equal(rows0, out_all[25:40])


def test_page_relabelling_invariance():
    """Moving pages to other indices (and the table with them) changes nothing."""
    spec = W.BatchSpec(hist=[19, 3], qlen=[6, 9], num_q_heads=2, num_kv_heads=1, head_dim=8,
                       page_size=4, seed=31, extra_pages=3)
    b = W.make_batch(spec)
    out, kc, vc = build_cache_and_run(b)
    perm = np.random.default_rng(5).permutation(b.num_pages)  # new index of old page i
    kc2 = np.empty_like(kc); vc2 = np.empty_like(vc)
    kc2[perm] = kc; vc2[perm] = vc
    bt2 = np.where(b.block_table >= 0, perm[np.maximum(b.block_table, 0)], -1).astype(np.int32)
    out2 = oracle.paged_attention(b.q, kc2, vc2, b.query_lens, b.seq_lens, bt2)
    assert np.array_equal(out, out2)


def test_dense_masked_softmax_cross_check_small_workload():
    """A dense fp64 masked-softmax formulation agrees on the small workload."""
    b = W.make_batch(W.spec_one_chunk_small())
    out, _, _ = build_cache_and_run(b)
    f = lambda x: W.bf16_bits_to_f32(x).astype(np.float64)
    K = np.concatenate([f(b.hist_k), f(b.k)])       # [384, 4, 64] positions 0..383
    V = np.concatenate([f(b.hist_v), f(b.v)])
    Q = f(b.q)                                     # [128, 4, 64] positions 256..383
    pos_q = 256 + np.arange(128)[:, None]
    mask = np.arange(384)[None, :] <= pos_q
    for h in range(4):
        S = Q[:, h, :] @ K[:, h, :].T / math.sqrt(64)
        S = np.where(mask, S, -np.inf)
        S -= S.max(axis=1, keepdims=True)
        E = np.exp(S)
        ref = (E / E.sum(axis=1, keepdims=True)) @ V[:, h, :]
        np.testing.assert_allclose(out[:, h, :], ref, rtol=0, atol=1e-12)


def test_kv_write_hand_placed_slots_and_sentinel():
    P, Hkv, d, pages = 2, 2, 2, 3
    k = np.arange(4 * Hkv * d, dtype=np.uint16).reshape(4, Hkv, d) + 1
    v = k + 100
    slots = np.array([5, 0, -1, 2], dtype=np.int64)  # page 2 off 1, page 0 off 0, padding, page 1 off 0
    kc = np.full((pages, Hkv, P, d), W.BF16_NAN_SENTINEL, dtype=np.uint16); vc = kc.copy()
    assert oracle.kv_cache_write(k, v, slots, P, kc, vc) == 0
    expect = np.full_like(kc, W.BF16_NAN_SENTINEL)
    for t, (pg, off) in {0: (2, 1), 1: (0, 0), 3: (1, 0)}.items():
        for h in range(Hkv):
            expect[pg, h, off, :] = k[t, h, :]
    assert np.array_equal(kc, expect)
    assert np.array_equal(vc[expect != W.BF16_NAN_SENTINEL], (expect + 100)[expect != W.BF16_NAN_SENTINEL])


def test_kv_write_out_of_range_slot_is_counted_and_skipped():
    k = np.ones((2, 1, 2), dtype=np.uint16); v = k.copy()
    kc = np.full((1, 1, 2, 2), W.BF16_NAN_SENTINEL, dtype=np.uint16); vc = kc.copy()
    assert oracle.kv_cache_write(k, v, np.array([1, 2]), 2, kc, vc) == 1
    assert np.all(kc[0, 0, 1] == 1) and np.all(kc[0, 0, 0] == W.BF16_NAN_SENTINEL)


def test_malformed_batch_is_rejected():
    b = W.make_batch(W.BatchSpec(hist=[2], qlen=[3], num_q_heads=1, num_kv_heads=1, head_dim=4,
                                 page_size=4, seed=1))
    kc = W.empty_cache(b); vc = W.empty_cache(b)
    with pytest.raises(ValueError):
        oracle.paged_attention(b.q, kc, vc, [4], [5], b.block_table)   # sum != T
    with pytest.raises(ValueError):
        oracle.paged_attention(b.q, kc, vc, [3], [2], b.block_table)   # seq < query


def test_bf16_rounding_of_the_generator():
    # ties to even and ordinary rounding, checked on hand-picked float32 values
    vals = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e-3], dtype=np.float32)
    bits = W.f32_to_bf16_bits(vals)
    assert bits[0] == 0x3F80
    assert bits[1] == 0x3F80          # 1 + 2^-8 is a tie -> even (down)
    assert bits[2] == 0x3F82          # 1 + 3*2^-8 is a tie -> even (up)
    assert bits[3] == 0xC020
    back = W.bf16_bits_to_f32(bits)
    assert abs(back[4] - 3.0e-3) <= 3.0e-3 * 2 ** -8
