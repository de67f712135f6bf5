"""Shared test helpers: move seeded batches to the GPU, run the library and the
oracle on the same inputs, and compare (no arithmetic of the method here)."""
from __future__ import annotations

import numpy as np

import oracle
import workloads as W

ATOL = 2e-2      # max-abs bound for attention (bf16 in, fp32 accumulate, bf16 out)
RTOL_F = 5e-3    # relative Frobenius bound


def to_dev_bf16(a, dev="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def to_dev(a, dev="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def bf16_tensor_to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def compare(got, ref, atol=ATOL, rtol_f=RTOL_F, what=""):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    diff = np.abs(got - ref)
    max_abs = float(diff.max()) if diff.size else 0.0
    nref = float(np.linalg.norm(ref))
    rel_f = float(np.linalg.norm(got - ref) / nref) if nref > 0 else float(np.linalg.norm(got - ref))
    assert max_abs <= atol and rel_f <= rtol_f, f"{what}: max-abs {max_abs:.3e} rel-F {rel_f:.3e}"
    return max_abs, rel_f


def oracle_caches(batch):
    kc = W.empty_cache(batch)
    vc = W.empty_cache(batch)
    P = batch.spec.page_size
    if batch.hist_k is not None and batch.hist_k.shape[0]:
        oracle.kv_cache_write(batch.hist_k, batch.hist_v, batch.hist_slot_mapping, P, kc, vc)
    oracle.kv_cache_write(batch.k, batch.v, batch.slot_mapping, P, kc, vc)
    return kc, vc


def run_gpu_batch(cpsa, batch, max_kv_splits=8, workspace_bytes=None, scale=0.0, block_table=None):
    """History and new tokens written by cpp_kv_cache_write into NaN-filled caches,
    then cpp_chunked_prefill_attn. Returns (out float64, flags, k_cache, v_cache)."""
    import torch
    s = batch.spec
    kc = to_dev(W.empty_cache(batch).view(np.int16)).view(torch.bfloat16)
    vc = kc.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if batch.hist_k is not None and batch.hist_k.shape[0]:
        cpsa.cpp_kv_cache_write(to_dev_bf16(batch.hist_k), to_dev_bf16(batch.hist_v),
                                to_dev(batch.hist_slot_mapping), kc, vc, err)
    T = batch.num_tokens
    if T:
        cpsa.cpp_kv_cache_write(to_dev_bf16(batch.k), to_dev_bf16(batch.v), to_dev(batch.slot_mapping), kc, vc, err)
    B = len(s.qlen)
    if workspace_bytes is None:
        workspace_bytes = cpsa.cpp_attn_workspace_bytes(B, T, s.num_q_heads, s.num_kv_heads, s.head_dim,
                                                        max_kv_splits)
    ws = torch.empty(workspace_bytes, dtype=torch.uint8, device="cuda")
    out = torch.full((T, s.num_q_heads, s.head_dim), float("nan"), dtype=torch.bfloat16, device="cuda")
    bt = batch.block_table if block_table is None else block_table
    cpsa.cpp_chunked_prefill_attn(to_dev_bf16(batch.q), kc, vc, to_dev(batch.query_lens), to_dev(batch.seq_lens),
                                  to_dev(bt), out, ws, err, scale=scale, max_kv_splits=max_kv_splits)
    torch.cuda.synchronize()
    flags = cpsa.cpp_read_device_error(err)
    return bf16_tensor_to_f64(out), flags, kc, vc


def run_gpu_batch_fused(cpsa, batch, max_kv_splits=8, scale=0.0, slot_mapping=None, workspace_bytes=None):
    """History written by cpp_kv_cache_write into NaN-filled caches, then one
    cpp_chunked_prefill_attn_write_kv call that writes the new tokens and attends.
    Returns (out float64, flags, k_cache, v_cache)."""
    import torch
    s = batch.spec
    kc = to_dev(W.empty_cache(batch).view(np.int16)).view(torch.bfloat16)
    vc = kc.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if batch.hist_k is not None and batch.hist_k.shape[0]:
        cpsa.cpp_kv_cache_write(to_dev_bf16(batch.hist_k), to_dev_bf16(batch.hist_v),
                                to_dev(batch.hist_slot_mapping), kc, vc, err)
    T = batch.num_tokens
    B = len(s.qlen)
    if workspace_bytes is None:
        workspace_bytes = cpsa.cpp_attn_workspace_bytes(B, T, s.num_q_heads, s.num_kv_heads, s.head_dim,
                                                        max_kv_splits)
    ws = torch.empty(workspace_bytes, dtype=torch.uint8, device="cuda")
    out = torch.full((T, s.num_q_heads, s.head_dim), float("nan"), dtype=torch.bfloat16, device="cuda")
    sm = batch.slot_mapping if slot_mapping is None else slot_mapping
    cpsa.cpp_chunked_prefill_attn_write_kv(to_dev_bf16(batch.q), to_dev_bf16(batch.k), to_dev_bf16(batch.v),
                                           to_dev(sm), kc, vc, to_dev(batch.query_lens), to_dev(batch.seq_lens),
                                           to_dev(batch.block_table), out, ws, err, scale=scale,
                                           max_kv_splits=max_kv_splits)
    torch.cuda.synchronize()
    flags = cpsa.cpp_read_device_error(err)
    return bf16_tensor_to_f64(out), flags, kc, vc


def cache_bits(t):
    """A bf16 device cache as uint16 bits on the host."""
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
