"""GPU parity of attention calls captured in a CUDA graph and replayed on new
inputs: a replay keeps the capture's sizes, pointers and per-call epoch, so
merge counters and partial results must not carry anything from one replay to
the next. Each case captures one call, then replays it on two batches of the
same lengths but different values (and page tables), each replay checked
against the fp64 oracle; a call outside the graph between replays must not
disturb them either."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import bf16_tensor_to_f64, compare, oracle_caches, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


class _Bufs:
    """Device buffers of one batch shape, refilled in place for each batch."""

    def __init__(self, torch, cpsa, b, max_kv_splits):
        s = b.spec
        T, B = b.num_tokens, len(s.qlen)
        self.q = to_dev_bf16(b.q)
        self.k = to_dev_bf16(b.k)
        self.v = to_dev_bf16(b.v)
        self.slots = to_dev(b.slot_mapping)
        self.kc = to_dev(W.empty_cache(b).view(np.int16)).view(torch.bfloat16)
        self.vc = self.kc.clone()
        self.ql = to_dev(b.query_lens)
        self.sl = to_dev(b.seq_lens)
        self.bt = to_dev(b.block_table)
        self.out = torch.empty((T, s.num_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
        self.ws = torch.empty(cpsa.cpp_attn_workspace_bytes(B, T, s.num_q_heads, s.num_kv_heads, s.head_dim,
                                                            max_kv_splits), dtype=torch.uint8, device="cuda")
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def load(self, torch, cpsa, b, fused):
        """Caches NaN-filled, the history written, the new rows written unless the
        call itself writes them; inputs and page table copied in place."""
        self.q.copy_(to_dev_bf16(b.q))
        self.k.copy_(to_dev_bf16(b.k))
        self.v.copy_(to_dev_bf16(b.v))
        self.slots.copy_(to_dev(b.slot_mapping))
        self.bt.copy_(to_dev(b.block_table))
        self.kc.copy_(to_dev(W.empty_cache(b).view(np.int16)).view(torch.bfloat16))
        self.vc.copy_(self.kc)
        self.out.fill_(float("nan"))
        if b.hist_k is not None and b.hist_k.shape[0]:
            cpsa.cpp_kv_cache_write(to_dev_bf16(b.hist_k), to_dev_bf16(b.hist_v), to_dev(b.hist_slot_mapping),
                                    self.kc, self.vc, self.err)
        if not fused:
            cpsa.cpp_kv_cache_write(self.k, self.v, self.slots, self.kc, self.vc, self.err)
        torch.cuda.synchronize()

    def call(self, cpsa, fused, max_kv_splits):
        if fused:
            cpsa.cpp_chunked_prefill_attn_write_kv(self.q, self.k, self.v, self.slots, self.kc, self.vc, self.ql,
                                                   self.sl, self.bt, self.out, self.ws, self.err,
                                                   max_kv_splits=max_kv_splits)
        else:
            cpsa.cpp_chunked_prefill_attn(self.q, self.kc, self.vc, self.ql, self.sl, self.bt, self.out, self.ws,
                                          self.err, max_kv_splits=max_kv_splits)


def _check(torch, cpsa, bufs, b, what):
    torch.cuda.synchronize()
    assert cpsa.cpp_read_device_error(bufs.err) == 0, what
    kc, vc = oracle_caches(b)
    ref = oracle.paged_attention(b.q, kc, vc, b.query_lens, b.seq_lens, b.block_table)
    compare(bf16_tensor_to_f64(bufs.out), ref, what=what)


CASES = {
    # one request: the chunk kernel plans its own runs; units cut across runs
    "self_planned_split": dict(hist=[9000], qlen=[512]),
    # several requests and decode rows: plan kernel, split decode rows (combine kernel)
    "planned_mixed": dict(hist=[6000, 0, 9000, 5000, 300], qlen=[384, 200, 1, 1, 1]),
    # more than 32 requests: the block-wide plan kernel
    "block_planned": dict(hist=[0, 0, 700] + [1000] * 30, qlen=[300, 300, 200] + [1] * 30),
}


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("case", sorted(CASES))
def test_graph_replay_new_inputs(cuda_lib, case, fused):
    import torch
    splits = 8
    specs = [W.BatchSpec(**CASES[case], num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                         seed=3100 + 10 * i + int(fused)) for i in range(3)]
    batches = [W.make_batch(s) for s in specs]
    bufs = _Bufs(torch, cuda_lib, batches[0], splits)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        bufs.load(torch, cuda_lib, batches[0], fused)
        bufs.call(cuda_lib, fused, splits)          # outside the graph: module loaded, attributes set
    torch.cuda.current_stream().wait_stream(side)
    _check(torch, cuda_lib, bufs, batches[0], f"{case} eager")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bufs.call(cuda_lib, fused, splits)
    for i, b in enumerate([batches[1], batches[2], batches[1]]):
        bufs.load(torch, cuda_lib, b, fused)
        g.replay()
        _check(torch, cuda_lib, bufs, b, f"{case} replay {i}")
        if i == 1:
            # an eager call (new epoch) between replays
            bufs.load(torch, cuda_lib, batches[0], fused)
            bufs.call(cuda_lib, fused, splits)
            _check(torch, cuda_lib, bufs, batches[0], f"{case} eager between replays")


def test_graph_replay_records_timing_marks(cuda_lib):
    """The timing-marks entry point captured in a graph: its marks become event
    nodes, readable after every replay, while the output still meets the oracle
    on the replay's own inputs."""
    import torch
    specs = [W.BatchSpec(hist=[9000], qlen=[512], num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                         seed=3300 + i) for i in range(2)]
    batches = [W.make_batch(s) for s in specs]
    bufs = _Bufs(torch, cuda_lib, batches[0], 8)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]

    def call():
        cuda_lib.cpp_chunked_prefill_attn_events(bufs.q, bufs.kc, bufs.vc, bufs.ql, bufs.sl, bufs.bt, bufs.out,
                                                 bufs.ws, bufs.err, ev, max_kv_splits=8)

    bufs.load(torch, cuda_lib, batches[0], False)
    call()
    torch.cuda.synchronize()
    t_stream = ev[1].elapsed_time(ev[2])
    # the chunk kernel of 512 queries over 9512 keys runs for tens of microseconds:
    # marks recorded back to back (not around the kernel) would read far less
    assert 0.01 < t_stream < 1000.0, t_stream
    _check(torch, cuda_lib, bufs, batches[0], "marks, stream launch")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    bufs.load(torch, cuda_lib, batches[1], False)
    g.replay()
    torch.cuda.synchronize()
    t_graph = ev[1].elapsed_time(ev[2])
    assert 0.01 < t_graph < 1000.0, t_graph
    _check(torch, cuda_lib, bufs, batches[1], "marks, graph replay")
