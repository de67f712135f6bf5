"""GPU parity of cpp_kv_cache_write against the oracle's KV write (bit-exact)."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _gpu_write(cpsa, batch, k, v, slots, kc_init=None):
    import torch
    kc = to_dev(W.empty_cache(batch).view(np.int16) if kc_init is None else kc_init.view(np.int16)).view(torch.bfloat16)
    vc = kc.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cpsa.cpp_kv_cache_write(to_dev_bf16(k), to_dev_bf16(v), to_dev(slots), kc, vc, err)
    torch.cuda.synchronize()
    return (kc.view(torch.int16).cpu().numpy().view(np.uint16), vc.view(torch.int16).cpu().numpy().view(np.uint16),
            cpsa.cpp_read_device_error(err))


@pytest.mark.parametrize("spec_fn", [
    lambda: W.spec_one_chunk_small(),
    lambda: W.BatchSpec(hist=[0, 5, 300, 17], qlen=[700, 1, 33, 250], num_q_heads=32, num_kv_heads=8,
                        head_dim=128, page_size=16, seed=41, extra_pages=9),
    lambda: W.BatchSpec(hist=[1000], qlen=[512], num_q_heads=8, num_kv_heads=8, head_dim=64,
                        page_size=128, seed=42, extra_pages=2),
    lambda: W.BatchSpec(hist=[3, 0], qlen=[9, 31], num_q_heads=2, num_kv_heads=1, head_dim=128,
                        page_size=8, seed=43),
])
def test_kv_write_bit_exact(cuda_lib, spec_fn):
    b = W.make_batch(spec_fn())
    gk, gv, flags = _gpu_write(cuda_lib, b, b.k, b.v, b.slot_mapping)
    ok, ov = W.empty_cache(b), W.empty_cache(b)
    oracle.kv_cache_write(b.k, b.v, b.slot_mapping, b.spec.page_size, ok, ov)
    assert flags == 0
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)


def test_kv_write_padding_and_out_of_range(cuda_lib):
    b = W.make_batch(W.BatchSpec(hist=[0], qlen=[64], num_q_heads=4, num_kv_heads=4, head_dim=64,
                                 page_size=16, seed=44, extra_pages=1))
    slots = b.slot_mapping.copy()
    slots[3] = -1                       # padding: skipped silently
    slots[10] = b.num_pages * 16        # out of range: skipped, flagged
    slots[11] = 10 ** 12
    gk, gv, flags = _gpu_write(cuda_lib, b, b.k, b.v, slots)
    ok, ov = W.empty_cache(b), W.empty_cache(b)
    assert oracle.kv_cache_write(b.k, b.v, slots, 16, ok, ov) == 2
    assert flags == cuda_lib.DEV_SLOT_OUT_OF_RANGE
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)


def test_kv_write_empty_call_is_ok(cuda_lib):
    import torch
    kc = torch.zeros((2, 1, 8, 64), dtype=torch.bfloat16, device="cuda")
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    k = torch.zeros((0, 1, 64), dtype=torch.bfloat16, device="cuda")
    cuda_lib.cpp_kv_cache_write(k, k, torch.zeros(0, dtype=torch.int64, device="cuda"), kc, kc.clone(), e)
    assert cuda_lib.cpp_read_device_error(e) == 0


def test_kv_write_rejects_bad_head_dim(cuda_lib):
    import torch
    kc = torch.zeros((2, 1, 8, 96), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 1, 96), dtype=torch.bfloat16, device="cuda")
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(cuda_lib.CpsaError):
        cuda_lib.cpp_kv_cache_write(k, k, torch.zeros(1, dtype=torch.int64, device="cuda"), kc, kc.clone(), e)


@pytest.mark.parametrize("which", ["sarathi_mixed", "microbatch"])
def test_kv_write_full_workloads_sampled_pages(cuda_lib, which):
    """Full-size batches; pages sampled, every token of a sampled page checked."""
    import torch
    spec = W.spec_sarathi_mixed() if which == "sarathi_mixed" else W.spec_microbatch()
    d = W.device_batch(spec)
    P, Hkv, D = spec.page_size, spec.num_kv_heads, spec.head_dim
    rng = np.random.default_rng(5)
    slots = d["slot_mapping_host"]
    pages_touched = np.unique(slots // P)
    pick = np.sort(rng.choice(pages_touched, size=min(256, len(pages_touched)), replace=False))
    pick_t = torch.from_numpy(pick).cuda()
    before_k = d["k_cache"][pick_t].view(torch.int16).cpu().numpy().view(np.uint16)
    before_v = d["v_cache"][pick_t].view(torch.int16).cpu().numpy().view(np.uint16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cuda_lib.cpp_kv_cache_write(d["k"], d["v"], d["slot_mapping"], d["k_cache"], d["v_cache"], err)
    torch.cuda.synchronize()
    assert cuda_lib.cpp_read_device_error(err) == 0
    after_k = d["k_cache"][pick_t].view(torch.int16).cpu().numpy().view(np.uint16)
    after_v = d["v_cache"][pick_t].view(torch.int16).cpu().numpy().view(np.uint16)
    # oracle on a compact cache holding only the sampled pages (prior contents as input)
    remap = {int(p): i for i, p in enumerate(pick)}
    sel = np.nonzero(np.isin(slots // P, pick))[0]
    cslots = np.array([remap[int(s // P)] * P + int(s % P) for s in slots[sel]], dtype=np.int64)
    k_host = d["k"][torch.from_numpy(sel).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
    v_host = d["v"][torch.from_numpy(sel).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
    ok, ov = before_k.copy(), before_v.copy()
    assert oracle.kv_cache_write(k_host, v_host, cslots, P, ok, ov) == 0
    assert ok.shape == (len(pick), Hkv, P, D)
    assert np.array_equal(after_k, ok) and np.array_equal(after_v, ov)
