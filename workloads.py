"""Seeded synthetic inputs for chunked-prefill paged attention.

This module only draws random numbers and lays them out in the input formats of
the library and the oracle. It holds none of the method's arithmetic: no
attention, no KV write, no split. Both `oracle/` (through the tests) and the
CUDA path (through the tests and `bench.py`) receive the same arrays from here.

Input recipe (one generator per workload, numpy PCG64 seeded per workload):

* values ~ N(0, 1) drawn in float32 and rounded to bf16 with round-to-nearest-even;
  bf16 is carried as uint16 bit patterns on the host;
* a request r has history h_r and query_len q_r; seq_len s_r = h_r + q_r
  (the new tokens are the last q_r of the s_r positions);
* the page pool is `rng.permutation(num_pages)`, handed out in request order, one
  page per `page_size` positions; unused block_table entries are -1;
* slot_mapping of position p of request r is `page * page_size + p % page_size`
  with `page = block_table[r][p // page_size]`, the slot format a serving
  scheduler hands to the KV write (the caches are `[num_pages, Hkv, P, d]`).

The large workloads (tens of GB of cache) draw their history directly into the
cache on the device with a seeded `torch.Generator`; see `device_cache_fill`.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BF16_NAN_SENTINEL = 0xFFFF  # a quiet-NaN bf16 pattern used to fill unwritten slots


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def randn_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


@dataclass
class BatchSpec:
    """One step's batch: per request history length and query length."""
    hist: list
    qlen: list
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    seed: int
    extra_pages: int = 0           # spare pages in the pool beyond the exact need
    name: str = ""

    @property
    def seq(self):
        return [h + q for h, q in zip(self.hist, self.qlen)]


@dataclass
class Batch:
    spec: BatchSpec
    q: np.ndarray            # uint16 [T, Hq, d]
    k: np.ndarray            # uint16 [T, Hkv, d]   new tokens' keys
    v: np.ndarray            # uint16 [T, Hkv, d]
    slot_mapping: np.ndarray  # int64 [T]
    block_table: np.ndarray   # int32 [B, max_blocks], -1 padded
    query_lens: np.ndarray    # int32 [B]
    seq_lens: np.ndarray      # int32 [B]
    num_pages: int
    hist_k: np.ndarray | None = None   # uint16 [sum h, Hkv, d] history keys (token-major)
    hist_v: np.ndarray | None = None
    hist_slot_mapping: np.ndarray | None = None  # int64 [sum h]
    extra: dict = field(default_factory=dict)

    @property
    def num_tokens(self):
        return int(self.q.shape[0])


def _pages_and_slots(spec: BatchSpec, rng: np.random.Generator):
    P = spec.page_size
    seq = spec.seq
    need = [(s + P - 1) // P for s in seq]
    num_pages = int(sum(need)) + int(spec.extra_pages)
    perm = rng.permutation(num_pages).astype(np.int64)
    max_blocks = max(1, max(need) if need else 1)
    bt = np.full((len(seq), max_blocks), -1, dtype=np.int32)
    cursor = 0
    for r, n in enumerate(need):
        bt[r, :n] = perm[cursor:cursor + n]
        cursor += n
    return bt, num_pages


def _slots_for(bt_row: np.ndarray, positions: np.ndarray, P: int) -> np.ndarray:
    pages = bt_row[positions // P].astype(np.int64)
    return pages * P + positions % P


def make_batch(spec: BatchSpec, with_history: bool = True) -> Batch:
    """Host (numpy) batch; history K/V returned token-major with its slot_mapping."""
    rng = np.random.Generator(np.random.PCG64(spec.seed))
    bt, num_pages = _pages_and_slots(spec, rng)
    P = spec.page_size
    T = int(sum(spec.qlen))
    H = int(sum(spec.hist))
    q = randn_bf16(rng, (T, spec.num_q_heads, spec.head_dim))
    k = randn_bf16(rng, (T, spec.num_kv_heads, spec.head_dim))
    v = randn_bf16(rng, (T, spec.num_kv_heads, spec.head_dim))
    slots = np.empty(T, dtype=np.int64)
    hslots = np.empty(H, dtype=np.int64)
    t = 0
    ht = 0
    for r, (h, ql) in enumerate(zip(spec.hist, spec.qlen)):
        slots[t:t + ql] = _slots_for(bt[r], np.arange(h, h + ql), P)
        hslots[ht:ht + h] = _slots_for(bt[r], np.arange(0, h), P)
        t += ql
        ht += h
    hist_k = hist_v = None
    if with_history:
        hist_k = randn_bf16(rng, (H, spec.num_kv_heads, spec.head_dim))
        hist_v = randn_bf16(rng, (H, spec.num_kv_heads, spec.head_dim))
    return Batch(spec=spec, q=q, k=k, v=v, slot_mapping=slots, block_table=bt,
                 query_lens=np.asarray(spec.qlen, dtype=np.int32),
                 seq_lens=np.asarray(spec.seq, dtype=np.int32),
                 num_pages=num_pages, hist_k=hist_k, hist_v=hist_v,
                 hist_slot_mapping=hslots)


def empty_cache(batch: Batch) -> np.ndarray:
    s = batch.spec
    return np.full((batch.num_pages, s.num_kv_heads, s.page_size, s.head_dim),
                   BF16_NAN_SENTINEL, dtype=np.uint16)


# ----------------------------------------------------------------------------
# The workloads (shapes of the pages' scenarios; values synthetic)
# ----------------------------------------------------------------------------

def spec_one_chunk_small(seed: int = 1) -> BatchSpec:
    """One request: history 256, chunk 128, 4/4 heads, d=64, page 16 (24 pages)."""
    return BatchSpec(hist=[256], qlen=[128], num_q_heads=4, num_kv_heads=4,
                     head_dim=64, page_size=16, seed=seed, name="one_chunk_h256_c128_d64")


LLAMA3_8B_HEADS = dict(num_q_heads=32, num_kv_heads=8, head_dim=128)


def spec_llama_chunk(history: int, chunk: int = 512, page_size: int = 128, seed: int = 2,
                     total_len: int = 32768) -> BatchSpec:
    """One chunk of a Llama-3-8B-shaped 32768-token prefill (32/8 heads, d=128).

    The page pool is the one of the whole 32768-token sequence, so the block_table
    is the same for every chunk."""
    spec = BatchSpec(hist=[history], qlen=[chunk], page_size=page_size, seed=seed,
                     name=f"llama_chunk_h{history}_c{chunk}", **LLAMA3_8B_HEADS)
    need_total = (total_len + page_size - 1) // page_size
    need_now = (history + chunk + page_size - 1) // page_size
    spec.extra_pages = max(0, need_total - need_now)
    return spec


def spec_sarathi_mixed(seed: int = 3, n_decode: int = 1536, ctx_lo: int = 1024,
                       ctx_hi: int = 8192, chunk: int = 512, chunk_hist: int = 8192,
                       page_size: int = 16) -> BatchSpec:
    """Token budget 2048: 1536 decode rows first, then one 512-token chunk at h=8192."""
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    ctx = rng.integers(ctx_lo, ctx_hi, size=n_decode, endpoint=True)
    hist = [int(c) - 1 for c in ctx] + [chunk_hist]
    qlen = [1] * n_decode + [chunk]
    return BatchSpec(hist=hist, qlen=qlen, page_size=page_size, seed=seed,
                     name="sarathi_mixed_budget2048", **LLAMA3_8B_HEADS)


def spec_microbatch(seed: int = 5, n_decode: int = 128, n_prefill: int = 64,
                    prompt: int = 2600, page_size: int = 16) -> BatchSpec:
    """128 decode rows (context U[2600, 5200]) then 64 fresh 2600-token prompts."""
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    ctx = rng.integers(prompt, 2 * prompt, size=n_decode, endpoint=True)
    hist = [int(c) - 1 for c in ctx] + [0] * n_prefill
    qlen = [1] * n_decode + [prompt] * n_prefill
    return BatchSpec(hist=hist, qlen=qlen, page_size=page_size, seed=seed,
                     name="microbatch_2600x64_plus_128dec", **LLAMA3_8B_HEADS)


def chunk_profile_sizes(base_chunk_size: int = 4096, n: int = 64):
    """The 64 profiling chunk sizes, uniform from base down toward 0: base*i/n."""
    return [base_chunk_size * i // n for i in range(1, n + 1)]


# ----------------------------------------------------------------------------
# Device-side generation for the large workloads (torch is plumbing here)
# ----------------------------------------------------------------------------

def device_batch(spec: BatchSpec, device="cuda"):
    """Same layout as `make_batch` but drawn on the device (torch RNG, seeded).

    Returns a dict of device tensors. History lives directly in the caches:
    every page is filled with N(0,1) bf16 drawn from the seeded generator, then
    the step's own tokens are written by the KV write under test."""
    import torch
    rng = np.random.Generator(np.random.PCG64(spec.seed))
    bt, num_pages = _pages_and_slots(spec, rng)
    P = spec.page_size
    T = int(sum(spec.qlen))
    slots = np.empty(T, dtype=np.int64)
    t = 0
    for r, (h, ql) in enumerate(zip(spec.hist, spec.qlen)):
        slots[t:t + ql] = _slots_for(bt[r], np.arange(h, h + ql), P)
        t += ql
    g = torch.Generator(device=device)
    g.manual_seed(spec.seed)
    bf = torch.bfloat16
    q = torch.randn((T, spec.num_q_heads, spec.head_dim), generator=g, device=device, dtype=torch.float32).to(bf)
    k = torch.randn((T, spec.num_kv_heads, spec.head_dim), generator=g, device=device, dtype=torch.float32).to(bf)
    v = torch.randn((T, spec.num_kv_heads, spec.head_dim), generator=g, device=device, dtype=torch.float32).to(bf)
    shape = (num_pages, spec.num_kv_heads, P, spec.head_dim)
    k_cache = torch.empty(shape, device=device, dtype=bf)
    v_cache = torch.empty(shape, device=device, dtype=bf)
    device_cache_fill(k_cache, g)
    device_cache_fill(v_cache, g)
    return dict(q=q, k=k, v=v,
                slot_mapping=torch.from_numpy(slots).to(device),
                block_table=torch.from_numpy(bt).to(device),
                query_lens=torch.tensor(spec.qlen, dtype=torch.int32, device=device),
                seq_lens=torch.tensor(spec.seq, dtype=torch.int32, device=device),
                k_cache=k_cache, v_cache=v_cache, num_pages=num_pages,
                block_table_host=bt, slot_mapping_host=slots)


def device_cache_fill(cache, gen, rows_per_fill: int = 1 << 14):
    """Fill a bf16 cache with N(0,1) in slabs (keeps the fp32 temporary small)."""
    import torch
    n = cache.shape[0]
    for p0 in range(0, n, rows_per_fill):
        p1 = min(n, p0 + rows_per_fill)
        slab = torch.randn(cache[p0:p1].shape, generator=gen, device=cache.device, dtype=torch.float32)
        cache[p0:p1].copy_(slab)
        del slab


def device_sequence(total_len: int = 32768, page_size: int = 128, num_q_heads: int = 32, num_kv_heads: int = 8,
                    head_dim: int = 128, seed: int = 2, device="cuda"):
    """One long prompt for chunked prefill: q/k/v of every position ~ N(0,1) bf16
    (seeded torch RNG on the device) and the slots of positions 0..total_len-1
    through a permuted pool of total_len / page_size pages.
    Returns (q, k, v, slot_mapping, block_table[1, pages]) device tensors."""
    import torch
    rng = np.random.Generator(np.random.PCG64(seed))
    n_pages = (total_len + page_size - 1) // page_size
    bt = rng.permutation(n_pages).astype(np.int32)[None, :]
    slots = _slots_for(bt[0], np.arange(total_len), page_size)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    bf = torch.bfloat16
    q = torch.randn((total_len, num_q_heads, head_dim), generator=g, device=device, dtype=torch.float32).to(bf)
    k = torch.randn((total_len, num_kv_heads, head_dim), generator=g, device=device, dtype=torch.float32).to(bf)
    v = torch.randn((total_len, num_kv_heads, head_dim), generator=g, device=device, dtype=torch.float32).to(bf)
    return q, k, v, torch.from_numpy(slots).to(device), torch.from_numpy(bt).to(device)
