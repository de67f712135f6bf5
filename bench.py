#!/usr/bin/env python
"""Benchmark of the chunked-prefill attention hot path on GB300.

Step = one pass of the whole path over the headline workload: a Llama-3-8B-shaped
attention layer (32 q / 8 kv heads, head_dim 128, bf16, page 128) prefilling one
32768-token sequence in 64 chunks of 512; per chunk the micro-batch split, the
slot_mapping KV write and the causal attention over the paged cache. The splits
run on a side stream joined back before the step ends (a one-request batch is
never split, so no attention call waits for one). The KV
write runs fused into the attention call (cpp_chunked_prefill_attn_write_kv);
`--two-call` times the separate write and attention calls instead, and the
line's `two_call_step` reports that variant on the same inputs. The step is
captured once in a CUDA graph and the graph is replayed for every timed step
(every kernel runs again on the resident inputs); `--eager` times stream
launches, and the line's `eager_step` reports them beside the graph.

Prints one JSON line (rank 0). `value` is attention TFLOP/s of the whole step
(algorithmic FLOPs: 4*d*Hq*sum_i (h + i + 1), unmasked pairs only) with inputs
resident in HBM; `e2e` is the same metric through the C ABI with host buffers
(pinned host->device copies of each chunk's q/k/v/slots and the device->host
read of its output inside the timed region, in the same launch mode, copies
included in the graph); `roofline` is the chunk kernel's
own event-timed throughput against the measured bf16 peak; `cpu_baseline` is
the fp64 oracle on a bounded sample of the same workload on the host cores.
`--impl reference` times that oracle alone on the workload's own metric.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

SEQ, CHUNK, HQ, HKV, D, PAGE = 32768, 512, 32, 8, 128, 128
N_CHUNKS = SEQ // CHUNK
E2E_BATCH = 4   # chunks per host<->device copy in the end-to-end measurement
WORKLOAD = "llama3-8b-attn-layer 32768-token prefill in 64 chunks of 512 (32/8 heads, d128, bf16, page 128)"
METRIC = "chunked-prefill attention TFLOP/s"


def chunk_flops(h, c, hq=HQ, d=D):
    """Algorithmic FLOPs of one chunk: QK^T and PV over the unmasked (query, key) pairs."""
    pairs = c * h + c * (c + 1) // 2
    return 4.0 * d * hq * pairs


STEP_FLOPS = sum(chunk_flops(i * CHUNK, CHUNK) for i in range(N_CHUNKS))


TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "chunk_attn_traffic_llama_chunked_prefill.md")
KERNEL_SOURCES = [os.path.join(ROOT, "chunked_prefill_paged_slot_gb300", "csrc", x)
                  for x in ("prefill_tc.cu", "common.cuh", "plan.cu", "plan.cuh")]


def source_code_only(text):
    """C/CUDA source with its comments removed and whitespace collapsed."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_digest():
    """sha256 over the chunk kernel's sources (the kernel and the plan that feeds it),
    comments and whitespace left out, so that only a change of code voids the
    recorded counters."""
    import hashlib
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "r") as f:
            h.update(source_code_only(f.read()).encode())
    return h.hexdigest()


def load_traffic():
    """DRAM bytes per chunk-kernel launch from the committed ncu summary, or None when
    the kernel's sources changed since those counters were taken."""
    try:
        fields = {}
        with open(TRAFFIC_PROFILE) as f:
            for ln in f:
                if ":" in ln and ln.strip().startswith("- "):
                    k, v = ln.strip()[2:].split(":", 1)
                    fields[k.strip()] = v.strip().strip("`")
        if fields.get("kernel_source_sha256") != kernel_source_digest():
            return None
        return float(fields["dram_bytes_per_launch"])
    except Exception:
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 6800.0, "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []          # (host time, csv line)
        self.window = (0.0, 0.0)

    def start(self):
        """Start sampling every 20 ms and wait (up to 5 s) until samples arrive."""
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "20"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
            return
        t0 = time.perf_counter()
        while not self.lines and time.perf_counter() - t0 < 5.0:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self, begin: float, end: float):
        """The timed region: only samples taken inside it are reported."""
        self.window = (begin, end)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        b, e = self.window
        for ts, ln in self.lines:
            if not (b <= ts <= e):
                continue
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- GPU workload
def draw_inputs(dev, seed=2):
    """Seeded inputs of the headline workload (see workloads.device_sequence)."""
    import workloads as W
    return W.device_sequence(SEQ, PAGE, HQ, HKV, D, seed=seed, device=dev)


class ChunkedPrefill:
    """Device buffers of the headline workload and its step."""

    def __init__(self, dev, seed=2, max_kv_splits=8, fused=True):
        import torch
        import chunked_prefill_paged_slot_gb300 as cpsa
        self.torch, self.cpsa, self.dev = torch, cpsa, dev
        self.fused = fused
        n_pages = SEQ // PAGE
        bf = torch.bfloat16
        self.q, self.k, self.v, self.slots, self.bt = draw_inputs(dev, seed)
        self.k_cache = torch.zeros((n_pages, HKV, PAGE, D), dtype=bf, device=dev)
        self.v_cache = torch.zeros_like(self.k_cache)
        self.out = torch.empty_like(self.q)
        self.qlens = torch.full((N_CHUNKS, 1), CHUNK, dtype=torch.int32, device=dev)
        self.slens = torch.tensor([[CHUNK * (i + 1)] for i in range(N_CHUNKS)], dtype=torch.int32, device=dev)
        self.max_kv_splits = max_kv_splits
        self.ws = torch.empty(cpsa.cpp_attn_workspace_bytes(1, CHUNK, HQ, HKV, D, max_kv_splits),
                              dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.split_outs = torch.zeros((N_CHUNKS, 3), dtype=torch.int32, device=dev)
        self.split_stream = torch.cuda.Stream(device=dev)
        self.marks = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(N_CHUNKS)]
        self.host = None

    def fork_splits(self, stream):
        """Start the side stream that computes the balanced micro-batch split of
        every chunk's batch (each result kept in split_outs). A one-request batch
        is never split, so no attention call waits for its split: the split runs
        beside the attention (its one warp fits next to a chunk-kernel CTA)
        rather than between the calls. chunk() enqueues chunk i's split just
        before its attention; join_splits() joins the side stream back."""
        fork = self.torch.cuda.Event()
        fork.record(stream)
        self.split_stream.wait_event(fork)

    def join_splits(self, stream):
        join = self.torch.cuda.Event()
        join.record(self.split_stream)
        stream.wait_event(join)

    def chunk(self, i, q, k, v, slots, out, stream, marks=None):
        cpsa = self.cpsa
        cpsa.cpp_split_microbatch(self.qlens[i], self.split_outs[i], 0.1, 256, stream=self.split_stream)
        if self.fused:
            cpsa.cpp_chunked_prefill_attn_write_kv(q, k, v, slots, self.k_cache, self.v_cache, self.qlens[i],
                                                   self.slens[i], self.bt, out, self.ws, self.err,
                                                   max_kv_splits=self.max_kv_splits, stream=stream,
                                                   events=None if marks is None else
                                                   [None, marks[0], marks[1], None, None])
            return
        cpsa.cpp_kv_cache_write(k, v, slots, self.k_cache, self.v_cache, self.err, stream=stream)
        if marks is None:
            cpsa.cpp_chunked_prefill_attn(q, self.k_cache, self.v_cache, self.qlens[i], self.slens[i], self.bt, out,
                                          self.ws, self.err, max_kv_splits=self.max_kv_splits, stream=stream)
        else:
            cpsa.cpp_chunked_prefill_attn_events(q, self.k_cache, self.v_cache, self.qlens[i], self.slens[i], self.bt,
                                                 out, self.ws, self.err, [None, marks[0], marks[1], None, None],
                                                 max_kv_splits=self.max_kv_splits, stream=stream)

    def step(self, stream, with_marks=False):
        self.fork_splits(stream)
        for i in range(N_CHUNKS):
            a, b = i * CHUNK, (i + 1) * CHUNK
            self.chunk(i, self.q[a:b], self.k[a:b], self.v[a:b], self.slots[a:b], self.out[a:b], stream,
                       self.marks[i] if with_marks else None)
        self.join_splits(stream)

    def chunk_kernel_ms(self):
        return [self.marks[i][0].elapsed_time(self.marks[i][1]) for i in range(N_CHUNKS)]

    # host-buffer variant for the end-to-end number: the step's inputs come from
    # pinned host memory and its output goes back there. Chunks are grouped in
    # batches of E2E_BATCH; each batch's inputs are copied in on one side stream
    # and its outputs copied out on another, into double buffers, so the copies
    # of batch b +- 1 overlap the attention of batch b. A plain torch kernel sits
    # between every cross-stream event and the library's kernels, so no event
    # operation is adjacent to a programmatically launched kernel.
    def make_host(self):
        torch = self.torch
        pin = lambda t: t.cpu().pin_memory()
        self.host = dict(q=pin(self.q), k=pin(self.k), v=pin(self.v), slots=pin(self.slots),
                         out=torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory())
        n = E2E_BATCH * CHUNK
        self.e2e_in = [dict(q=torch.empty((n, HQ, D), dtype=torch.bfloat16, device=self.dev),
                            k=torch.empty((n, HKV, D), dtype=torch.bfloat16, device=self.dev),
                            v=torch.empty((n, HKV, D), dtype=torch.bfloat16, device=self.dev),
                            slots=torch.empty(n, dtype=torch.int64, device=self.dev)) for _ in range(2)]
        self.e2e_out = [torch.empty((n, HQ, D), dtype=torch.bfloat16, device=self.dev) for _ in range(2)]
        self.e2e_streams = (torch.cuda.Stream(device=self.dev), torch.cuda.Stream(device=self.dev))
        self.e2e_tick = torch.zeros(1, dtype=torch.int32, device=self.dev)
        h2d = (self.q.numel() + self.k.numel() + self.v.numel()) * 2 + self.slots.numel() * 8
        return h2d, self.out.numel() * 2

    def step_e2e(self, stream):
        torch, h = self.torch, self.host
        s_in, s_out = self.e2e_streams
        nb = N_CHUNKS // E2E_BATCH
        ev = lambda: torch.cuda.Event()
        self.fork_splits(stream)
        start = ev()
        start.record(stream)
        h2d_done, comp_done, d2h_done = [None] * nb, [None] * nb, [None] * nb
        for b in range(nb):
            buf, out = self.e2e_in[b % 2], self.e2e_out[b % 2]
            a0, a1 = b * E2E_BATCH * CHUNK, (b + 1) * E2E_BATCH * CHUNK
            # inputs of batch b, once batch b - 2 (same buffers) has been computed
            s_in.wait_event(start if b < 2 else comp_done[b - 2])
            with torch.cuda.stream(s_in):
                for name in ("q", "k", "v", "slots"):
                    buf[name].copy_(h[name][a0:a1], non_blocking=True)
            h2d_done[b] = ev()
            h2d_done[b].record(s_in)
            # attention of batch b, once its inputs are in and batch b - 2's outputs are out
            stream.wait_event(h2d_done[b])
            if b >= 2:
                stream.wait_event(d2h_done[b - 2])
            with torch.cuda.stream(stream):
                self.e2e_tick.add_(1)
            for j in range(E2E_BATCH):
                i = b * E2E_BATCH + j
                sl = slice(j * CHUNK, (j + 1) * CHUNK)
                self.chunk(i, buf["q"][sl], buf["k"][sl], buf["v"][sl], buf["slots"][sl], out[sl], stream)
            with torch.cuda.stream(stream):
                self.e2e_tick.add_(1)
            comp_done[b] = ev()
            comp_done[b].record(stream)
            # outputs of batch b
            s_out.wait_event(comp_done[b])
            with torch.cuda.stream(s_out):
                h["out"][a0:a1].copy_(out, non_blocking=True)
            d2h_done[b] = ev()
            d2h_done[b].record(s_out)
        stream.wait_event(d2h_done[nb - 1])
        stream.wait_event(d2h_done[nb - 2])
        self.join_splits(stream)


# ----------------------------------------------------------------------------- oracle (CPU) leg
def oracle_sample(q, k, v, slots, bt, rows_per_chunk, rng, chunks=None):
    """Run the fp64 oracle on sampled rows of the workload; returns (seconds, flops, rows)."""
    import oracle
    import workloads as W
    n_pages = SEQ // PAGE
    kc = np.full((n_pages, HKV, PAGE, D), W.BF16_NAN_SENTINEL, dtype=np.uint16)
    vc = kc.copy()
    oracle.kv_cache_write(k, v, slots, PAGE, kc, vc)   # whole sequence cached (history of every chunk)
    chunks = range(N_CHUNKS) if chunks is None else chunks
    total_s, flops, n = 0.0, 0.0, 0
    for i in chunks:
        h = i * CHUNK
        rows = np.sort(rng.choice(CHUNK, size=rows_per_chunk, replace=False))
        t0 = time.perf_counter()
        oracle.paged_attention(q[h:h + CHUNK], kc, vc, [CHUNK], [h + CHUNK], bt, rows=rows)
        total_s += time.perf_counter() - t0
        flops += sum(4.0 * D * HQ * (h + int(r) + 1) for r in rows)
        n += len(rows)
    return total_s, flops, n


def host_inputs(seed=2):
    """Host copies (uint16 bit patterns) of the workload's inputs, drawn on the device."""
    import torch
    q, k, v, slots, bt = draw_inputs(torch.device("cuda"), seed)
    to16 = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    return (to16(q), to16(k), to16(v), slots.cpu().numpy(), bt.cpu().numpy())


def cpu_baseline(inputs, budget_s=12.0):
    import oracle
    q, k, v, slots, bt = inputs
    rng = np.random.default_rng(0)
    # calibrate on one row of the last chunk, then size the sample to ~budget_s
    s1, f1, _ = oracle_sample(q, k, v, slots, bt, 1, rng, chunks=[N_CHUNKS - 1])
    per_flop = s1 / f1
    avg_row_flops = STEP_FLOPS / SEQ
    rows_per_chunk = int(max(1, min(CHUNK, budget_s / (per_flop * avg_row_flops * N_CHUNKS))))
    s, f, n = oracle_sample(q, k, v, slots, bt, rows_per_chunk, rng)
    return {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} query rows ({rows_per_chunk} per chunk, all 32 heads) across the 64 chunks; "
                      f"{f / 1e9:.1f} GFLOP fp64 in {s:.1f} s"}


# ----------------------------------------------------------------------------- secondary: decode bandwidth
def decode_bandwidth(dev, reps=5, n_decode=1536):
    """Decode-row HBM GB/s on the Sarathi mixed step (n_decode decode rows + one 512 chunk at h=8192)."""
    import torch
    import chunked_prefill_paged_slot_gb300 as cpsa
    import workloads as W
    spec = W.spec_sarathi_mixed(n_decode=n_decode)
    d = W.device_batch(spec, device=dev)
    B, T = len(spec.qlen), sum(spec.qlen)
    ws = torch.empty(cpsa.cpp_attn_workspace_bytes(B, T, HQ, HKV, D, 8), dtype=torch.uint8, device=dev)
    out = torch.empty_like(d["q"])
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    cpsa.cpp_kv_cache_write(d["k"], d["v"], d["slot_mapping"], d["k_cache"], d["v_cache"], err)
    dec_ms, chunk_ms, step_ms = [], [], []
    for r in range(reps + 2):
        flush.zero_()
        cpsa.cpp_chunked_prefill_attn_events(d["q"], d["k_cache"], d["v_cache"], d["query_lens"], d["seq_lens"],
                                             d["block_table"], out, ws, err, ev, max_kv_splits=8)
        torch.cuda.synchronize()
        if r >= 2:
            chunk_ms.append(ev[1].elapsed_time(ev[2]))
            dec_ms.append(ev[2].elapsed_time(ev[3]))
            step_ms.append(ev[0].elapsed_time(ev[4]))
    flags = cpsa.cpp_read_device_error(err)
    n_dec = sum(1 for x in spec.qlen if x == 1)
    ctx = np.array(spec.seq[:n_dec], dtype=np.float64)
    dec_bytes = float(ctx.sum()) * HKV * D * 2 * 2 + n_dec * HQ * D * 2 * 2
    chunk_f = chunk_flops(spec.hist[-1], spec.qlen[-1])
    res = {"workload": f"sarathi mixed step: {n_decode} decode rows (context U[1024,8192]) + one 512-token chunk "
                       "at h=8192, 32/8 heads, d128, page 16, L2 flushed",
           "decode_kernel_ms": float(np.median(dec_ms)),
           "decode_hbm_gbs": dec_bytes / (np.median(dec_ms) * 1e-3) / 1e9,
           "decode_bytes": dec_bytes,
           "chunk_kernel_ms": float(np.median(chunk_ms)),
           "chunk_tflops": chunk_f / (np.median(chunk_ms) * 1e-3) / 1e12,
           "attn_call_ms": float(np.median(step_ms)), "device_flags": flags}
    del d, ws, out, flush
    torch.cuda.empty_cache()
    return res


def kv_write_bandwidth(dev, reps=5):
    """KV write GB/s (algorithmic bytes 2*T*Hkv*d*2*2 + 8T: read k and v, write both
    caches, read the slots) for the headline chunk (T = 512, page 128) and for the
    micro-batch workload's token count (T = 166528, page 16), slots a permutation of
    the cache's slots, L2 flushed before each repetition."""
    import torch
    import chunked_prefill_paged_slot_gb300 as cpsa
    res = {}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    for T, P in ((CHUNK, PAGE), (166528, 16)):
        n_pages = (T + P - 1) // P
        k = torch.randn((T, HKV, D), generator=g, device=dev).to(torch.bfloat16)
        v = torch.randn((T, HKV, D), generator=g, device=dev).to(torch.bfloat16)
        kc = torch.empty((n_pages, HKV, P, D), dtype=torch.bfloat16, device=dev)
        vc = torch.empty_like(kc)
        slots = torch.randperm(n_pages * P, generator=g, device=dev)[:T].to(torch.int64)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts = []
        for r in range(reps + 2):
            flush.zero_()
            e0.record()
            cpsa.cpp_kv_cache_write(k, v, slots, kc, vc, err)
            e1.record()
            torch.cuda.synchronize()
            if r >= 2:
                ts.append(e0.elapsed_time(e1))
        ms = float(np.median(ts))
        nbytes = 2.0 * T * HKV * D * 2 * 2 + 8 * T
        res[f"T{T}_page{P}"] = {"ms": round(ms, 4), "bytes": nbytes, "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}
        del k, v, kc, vc, slots
    res["device_flags"] = cpsa.cpp_read_device_error(err)
    del flush
    torch.cuda.empty_cache()
    return res


def serving_loop(dev, chunk_caps=(), tile_align=0, budget=2048, n_req=32, decode_tokens=32, seed=11, fused=False):
    """Closed loop: the library's token-budget batch builder sizes every step
    (decode rows first, then started prompts, then new ones) and allocates pages;
    each step runs the KV write and the attention kernels on it. Llama-3-8B
    shapes (32/8 heads, d128), page 16, prompts U[512, 4096], `decode_tokens`
    decode rows per request. Device time per step from CUDA events around each
    call (host work inside the call included), and the whole loop again as one
    graph per step replayed back to back (the kernels' own time)."""
    import torch
    import chunked_prefill_paged_slot_gb300 as cpsa
    rng = np.random.Generator(np.random.PCG64(seed))
    prompts = rng.integers(512, 4096, size=n_req, endpoint=True)
    P = 16
    pages = int(sum((int(L) + decode_tokens + P - 1) // P for L in prompts)) + 64
    sched = cpsa.BatchScheduler(budget, P, pages, page_order=rng.permutation(pages).astype(np.int32),
                                chunk_caps=chunk_caps, tile_align=tile_align, max_reqs=256,
                                max_blocks=(4096 + decode_tokens) // P + 2)
    for i, L in enumerate(prompts):
        sched.add_request(i, int(L), decode_tokens)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    qp = torch.randn((budget, HQ, D), generator=g, device=dev).to(torch.bfloat16)
    kp = torch.randn((budget, HKV, D), generator=g, device=dev).to(torch.bfloat16)
    vp = torch.randn((budget, HKV, D), generator=g, device=dev).to(torch.bfloat16)
    kc = torch.zeros((pages, HKV, P, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    out = torch.empty((budget, HQ, D), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(cpsa.cpp_attn_workspace_bytes(256, budget, HQ, HKV, D, 8), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    evs, calls, prefill_tok, decode_tok, flops, steps = [], [], 0, 0, 0.0, 0
    t0 = time.perf_counter()
    while True:
        waiting, running, _, _ = sched.stats()
        if waiting == 0 and running == 0:
            break
        b = sched.step()
        B, T = len(b["req_ids"]), len(b["slot_mapping"])
        if B == 0:
            raise RuntimeError("serving loop made no progress")
        ql, sl = b["query_lens"], b["seq_lens"]
        meta = [torch.from_numpy(x).to(dev, non_blocking=True) for x in (ql, sl, b["block_table"], b["slot_mapping"])]
        def call(T=T, meta=meta, s=stream):
            if fused:
                cpsa.cpp_chunked_prefill_attn_write_kv(qp[:T], kp[:T], vp[:T], meta[3], kc, vc, meta[0], meta[1],
                                                       meta[2], out[:T], ws, err, max_kv_splits=8, stream=s)
            else:
                cpsa.cpp_kv_cache_write(kp[:T], vp[:T], meta[3], kc, vc, err, stream=s)
                cpsa.cpp_chunked_prefill_attn(qp[:T], kc, vc, meta[0], meta[1], meta[2], out[:T], ws, err,
                                              max_kv_splits=8, stream=s)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        evs.append((e0, e1))
        calls.append(call)
        dec = ql == 1
        decode_tok += int(dec.sum())
        prefill_tok += int(ql[~dec].sum())
        for q_r, s_r in zip(ql.tolist(), sl.tolist()):
            h_r = s_r - q_r
            flops += 4.0 * D * HQ * (q_r * h_r + q_r * (q_r + 1) // 2)
        sched.commit()
        steps += 1
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    ms = [a.elapsed_time(b_) for a, b_ in evs]
    # the same steps again, each captured in a graph of its own and replayed back
    # to back: the kernels' time without the host work between and inside the calls
    # (each step rewrites the same cache slots with the same rows)
    graphs = []
    cap = torch.cuda.Stream(device=dev)
    for call in calls:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=cap):
            call(s=cap)
        graphs.append(gr)
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for gr in graphs:
        gr.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    graph_ms = g0.elapsed_time(g1)
    del graphs
    flags = cpsa.cpp_read_device_error(err)
    sched.close()
    del kc, vc, qp, kp, vp, ws
    torch.cuda.empty_cache()
    return {"steps": steps, "prompt_tokens": prefill_tok, "decode_tokens": decode_tok,
            "device_ms": round(float(sum(ms)), 3), "mean_step_ms": round(float(np.mean(ms)), 4),
            "max_step_ms": round(float(np.max(ms)), 4), "wall_s": round(wall, 3),
            "tokens_per_s_device": round((prefill_tok + decode_tok) / (sum(ms) * 1e-3), 1),
            "attention_tflops_device": round(flops / (sum(ms) * 1e-3) / 1e12, 2),
            "graph_replay_ms": round(graph_ms, 3),
            "attention_tflops_graph_replay": round(flops / (graph_ms * 1e-3) / 1e12, 2), "device_flags": flags}


def step_roofline(ms_per_step, peak_tf, peak_gbs):
    """t_roof of the headline step: per chunk max(F / peak_bf16, bytes_attn / BW) plus the KV
    write's bytes / BW, bytes_attn = K and V of the chunk's keys once per kv head + q read and
    out written + the block_table entries."""
    t, tensor_bound = 0.0, 0
    for i in range(N_CHUNKS):
        s = (i + 1) * CHUNK
        f = chunk_flops(i * CHUNK, CHUNK)
        b_attn = s * HKV * D * 2 * 2 + 2 * CHUNK * HQ * D * 2 + 4 * ((s + PAGE - 1) // PAGE)
        b_kvw = 2 * CHUNK * HKV * D * 2 * 2 + 8 * CHUNK
        tf, tb = f / (peak_tf * 1e12), b_attn / (peak_gbs * 1e9)
        tensor_bound += tf >= tb
        t += max(tf, tb) + b_kvw / (peak_gbs * 1e9)
    return {"t_roof_ms": round(t * 1e3, 4), "frac": round(t * 1e3 / ms_per_step, 4),
            "chunks_tensor_bound": int(tensor_bound), "chunks": N_CHUNKS}


# ----------------------------------------------------------------------------- suite of the other workloads
class ChunkTimer:
    """Times one chunk (split + KV write + attention) of the headline sequence at
    any (history, chunk size) with CUDA events; L2 flushed before each repetition."""

    def __init__(self, dev):
        import torch
        import chunked_prefill_paged_slot_gb300 as cpsa
        self.torch, self.cpsa, self.dev = torch, cpsa, dev
        self.q, self.k, self.v, self.slots, self.bt = draw_inputs(dev)
        n_pages = SEQ // PAGE
        self.k_cache = torch.zeros((n_pages, HKV, PAGE, D), dtype=torch.bfloat16, device=dev)
        self.v_cache = torch.zeros_like(self.k_cache)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.split_out = torch.zeros(3, dtype=torch.int32, device=dev)
        self.ws = torch.empty(cpsa.cpp_attn_workspace_bytes(1, 8192, HQ, HKV, D, 8), dtype=torch.uint8, device=dev)
        self.out = torch.empty_like(self.q)
        self.flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        # the whole sequence's K/V in the cache (history of any chunk)
        for a in range(0, SEQ, 4096):
            cpsa.cpp_kv_cache_write(self.k[a:a + 4096], self.v[a:a + 4096], self.slots[a:a + 4096],
                                    self.k_cache, self.v_cache, self.err)
        torch.cuda.synchronize()

    def time(self, h, c, reps=5):
        torch, cpsa = self.torch, self.cpsa
        ql = torch.tensor([c], dtype=torch.int32, device=self.dev)
        sl = torch.tensor([h + c], dtype=torch.int32, device=self.dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts = []
        for r in range(reps + 2):
            self.flush.zero_()
            e0.record()
            cpsa.cpp_split_microbatch(ql, self.split_out, 0.1, 256)
            cpsa.cpp_kv_cache_write(self.k[h:h + c], self.v[h:h + c], self.slots[h:h + c], self.k_cache,
                                    self.v_cache, self.err)
            cpsa.cpp_chunked_prefill_attn(self.q[h:h + c], self.k_cache, self.v_cache, ql, sl, self.bt,
                                          self.out[h:h + c], self.ws, self.err, max_kv_splits=8)
            e1.record()
            torch.cuda.synchronize()
            if r >= 2:
                ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))


def fit_report(X, t):
    X = np.asarray(X, dtype=np.float64)
    t = np.asarray(t, dtype=np.float64)
    coef, *_ = np.linalg.lstsq(X, t, rcond=None)
    res = t - X @ coef
    return [float(c) for c in coef], {"rms_ms": float(np.sqrt(np.mean(res ** 2))),
                                      "max_rel": float(np.max(np.abs(res) / t))}


def suite(dev):
    """Dynamic chunking (profile, fit, plan, per-chunk times), the online-calibrated
    controller, the two-variable latency fit, tile alignment, and the micro-batch
    workload on one vs two streams."""
    import torch
    import chunked_prefill_paged_slot_gb300 as cpsa
    import workloads as W
    out = {}
    ct = ChunkTimer(dev)
    # --- profile: 64 sizes base*i/64 at history 0, fit f(l) = a l^2 + b l + c
    sizes = W.chunk_profile_sizes(4096, 64)
    prof = [ct.time(0, l, reps=3) for l in sizes]
    a, b, c = cpsa.cpp_fit_latency_quadratic(sizes, prof)
    _, fr = fit_report(np.stack([np.square(sizes), sizes, np.ones(len(sizes))], 1), prof)
    chunks = cpsa.cpp_plan_chunk_sizes(a, b, c, SEQ, 4096, PAGE, 64, 0, 0, 1.0)
    L = 0
    dyn = []
    for x in chunks:
        dyn.append(ct.time(L, x, reps=3))
        L += x
    body = dyn[:-1] if len(dyn) > 2 else dyn
    out["dynamic_chunks"] = {
        "workload": "32768-token prompt, chunk sizes from the solver on f(l) fitted to 64 profile sizes "
                    "l = 64..4096 at history 0 (page 128, min 64, base 4096, smoothing 1)",
        "fit_f_l": {"a": a, "b": b, "c": c, **fr}, "target_ms": a * 4096 ** 2 + b * 4096,
        "chunks": chunks, "chunk_ms": [round(v, 4) for v in dyn],
        "cv_excluding_last": float(np.std(body) / np.mean(body)), "total_ms": float(np.sum(dyn))}
    # --- online calibration: chunk sizes from the controller, fed back with each chunk's own time
    oc = cpsa.OnlineChunker(a, b, c, 4096, PAGE, min_chunk=64, window=30, min_points=5)
    L, och, oms = 0, [], []
    while L < SEQ:
        x = oc.next_chunk(L, SEQ - L)
        t_ms = ct.time(L, x, reps=3)
        oc.record([x], [L], t_ms)
        och.append(x)
        oms.append(t_ms)
        L += x
    (oa, ob, occ), n_rec, calibrated = oc.model()
    oc.close()
    obody = oms[:-1] if len(oms) > 2 else oms
    out["online_calibration"] = {
        "workload": "the same prompt, each next chunk from the online controller (startup model above, "
                    "two-variable refit over the last 30 chunks from the 5th on), fed each chunk's measured time",
        "chunks": och, "chunk_ms": [round(v, 4) for v in oms],
        "cv_excluding_last": float(np.std(obody) / np.mean(obody)), "total_ms": float(np.sum(oms)),
        "final_model": {"a": oa, "b": ob, "c": occ, "batches": n_rec, "calibrated": calibrated}}
    # --- fixed 512 chunks (the headline sequence) for f(C, H)
    fixed = [ct.time(512 * i, 512, reps=3) for i in range(N_CHUNKS)]
    samples_C = [512] * N_CHUNKS + list(chunks) + list(sizes)
    hs, L = [], 0
    for x in chunks:
        hs.append(L)
        L += x
    samples_H = [512 * i for i in range(N_CHUNKS)] + hs + [0] * len(sizes)
    times = fixed + dyn + prof
    Cs = np.asarray(samples_C, dtype=np.float64)
    Hs = np.asarray(samples_H, dtype=np.float64)
    a2, b2, c2 = cpsa.cpp_fit_latency_two_var(Cs * (Cs + Hs), Cs + Hs, np.ones_like(Cs), times)
    _, fr2 = fit_report(np.stack([Cs * (Cs + Hs), Cs + Hs, np.ones_like(Cs)], 1), times)
    out["fixed_chunks_512"] = {"chunk_ms": [round(v, 4) for v in fixed], "total_ms": float(np.sum(fixed))}
    out["fit_f_C_H"] = {"a": a2, "b": b2, "c": c2, "samples": len(times), **fr2}
    # --- tile alignment around 512 at history 8192
    out["tile_alignment_h8192"] = {str(x): round(ct.time(8192, x, reps=5), 4) for x in (511, 512, 513)}
    del ct
    torch.cuda.empty_cache()
    # --- closed-loop serving: batch builder + kernels, fixed chunks vs the progressive strategy
    out["serving_loop"] = {
        "workload": "32 requests, prompts U[512, 4096], 32 decode rows each, token budget 2048, page 16, "
                    "32/8 heads d128; every step sized by the library's batch builder; KV write and "
                    "attention as two calls (the fused call is timed beside it)",
        "budget_only": serving_loop(dev),
        "progressive_2048_1024_512": serving_loop(dev, chunk_caps=(2048, 1024, 512)),
        "budget_tile_128": serving_loop(dev, tile_align=128),
        "budget_only_fused_kv_write": serving_loop(dev, fused=True)}
    out["microbatch_two_streams"] = microbatch(dev)
    return out


def microbatch(dev, reps=5):
    """The micro-batch workload on one stream and on two (the balanced split), as
    two calls and with the KV write fused."""
    import torch
    import chunked_prefill_paged_slot_gb300 as cpsa
    import workloads as W
    spec = W.spec_microbatch()
    d = W.device_batch(spec, device=dev)
    B, T = len(spec.qlen), sum(spec.qlen)
    step = cpsa.AttentionStep(B, T, HQ, HKV, D, max_kv_splits=8, two_stream=True, device=dev)
    step_f = cpsa.AttentionStep(B, T, HQ, HKV, D, max_kv_splits=8, two_stream=True, device=dev,
                                fused_kv_write=True)
    o = torch.empty_like(d["q"])
    args = (d["q"], d["k"], d["v"], d["slot_mapping"], d["k_cache"], d["v_cache"], d["query_lens"],
            d["seq_lens"], d["block_table"], o)

    def timed(fn):
        """Median of (device ms between CUDA events on the calling stream, host wall
        ms around the same call, both synchronised). Both micro-batches' streams
        join the calling stream before its end event. The inputs (1.4 GB of q
        alone) exceed L2, so nothing is flushed between repetitions."""
        cur = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dv, hw = [], []
        for r in range(reps + 2):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            e0.record(cur)
            fn()
            e1.record(cur)
            torch.cuda.synchronize()
            if r >= 2:
                hw.append(1e3 * (time.perf_counter() - t0))
                dv.append(e0.elapsed_time(e1))
        return float(np.median(dv)), float(np.median(hw))
    one, one_wall = timed(lambda: step.run(*args))
    one_f, one_f_wall = timed(lambda: step_f.run(*args))
    # the split depends on the batch's lengths alone: the split kernel runs once
    # per batch, its result read back before the timed steps
    split = step.split(d["query_lens"])
    two, two_wall = timed(lambda: step.run_two_stream(*args, split=split))
    two_f, _ = timed(lambda: step_f.run_two_stream(*args, split=split))
    two_with_split, _ = timed(lambda: step.run_two_stream(*args))
    pf = sum(4.0 * D * HQ * (q * h + q * (q + 1) // 2) for q, h in zip(spec.qlen, spec.hist) if q > 1)
    tf = lambda ms: pf / (ms * 1e-3) / 1e12
    res = {
        "workload": "128 decode rows (context U[2600,5200]) + 64 prompts of 2600 tokens, page 16; "
                    "device time between CUDA events on the calling stream (host wall time beside it)",
        "split": list(step.last_split), "one_stream_ms": one, "two_streams_ms": two, "two_vs_one": two / one,
        "two_streams_with_split_readback_ms": two_with_split, "prefill_tflops_one_stream": tf(one),
        "fused_kv_write": {"one_stream_ms": one_f, "two_streams_ms": two_f, "two_vs_one": two_f / one_f,
                           "prefill_tflops_one_stream": tf(one_f)},
        "host_wall_ms": {"one_stream": one_wall, "two_streams": two_wall, "one_stream_fused": one_f_wall},
        "tokens_per_s_one_stream": T / (one * 1e-3), "device_flags": step.read_errors() | step_f.read_errors()}
    del d, step, step_f, o
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------- replicas
def max_over_ranks(x, dist, dev):
    """The largest value of x over all ranks (the slowest replica sets the job's
    time); x itself when there is no process group."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, flops_per_replica_step, steps, total_ms):
    """Whole-job TFLOP/s: each of the `world` replicas does one step's FLOPs per
    step, and the job takes the slowest replica's `total_ms` for `steps` steps."""
    return world * flops_per_replica_step * steps / (total_ms * 1e-3) / 1e12


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-suite", action="store_true")
    ap.add_argument("--no-compare", action="store_true",
                    help="skip timing the other variant of the step (for profiling runs)")
    ap.add_argument("--two-call", action="store_true",
                    help="time the KV write and the attention as two calls (default: the fused call)")
    ap.add_argument("--profile-decode", action="store_true",
                    help="only the mixed decode step with 128 decode rows (about 2.5 GB of cache), timed with "
                         "CUDA events; an ncu --set full capture of this case once ended in a GPU fault (see the "
                         "design notes on measurement) and is not to be repeated")
    ap.add_argument("--eager", action="store_true",
                    help="time the step as stream launches (default: one step, all 64 chunks and the side-stream "
                         "splits, captured once in a CUDA graph and replayed; the stream-launch step is then "
                         "timed beside it as eager_step)")
    ap.add_argument("--profile-kv-write", action="store_true",
                    help="only the KV-write bandwidth measurement (T = 512 at page 128, T = 166528 at page 16)")
    ap.add_argument("--profile-microbatch", action="store_true",
                    help="only the micro-batch workload (one and two streams, two calls and fused), each variant "
                         "run three times (one timed), for a launch list of its kernels")
    args = ap.parse_args()
    if args.profile_microbatch:
        import torch
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps(microbatch(dev, reps=1)), flush=True)
        return 0
    if args.profile_kv_write:
        import torch
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps(kv_write_bandwidth(dev, reps=3)), flush=True)
        return 0
    if args.profile_decode:
        import torch
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps(decode_bandwidth(dev, reps=3, n_decode=128)), flush=True)
        return 0
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return reference_arm(args, world, rank)

    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import chunked_prefill_paged_slot_gb300 as cpsa
    cpsa.load()

    wl = ChunkedPrefill(dev, fused=not args.two_call)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # > L2 (129 MB)
    for _ in range(max(3, args.warmup)):
        wl.step(stream)
    torch.cuda.synchronize()
    if cpsa.cpp_read_device_error(wl.err) != 0:
        raise SystemExit("device error flags set during warm-up")

    gpu_uuid = None
    try:
        gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
        gpu_uuid = gpu_uuid if gpu_uuid.startswith("GPU-") else "GPU-" + gpu_uuid
    except Exception:
        pass
    eager_step = lambda: wl.step(stream)
    run_step = eager_step
    if not args.eager:
        # the same step, captured once: the library's calls launch from the capture
        graph = torch.cuda.CUDAGraph()
        capture = torch.cuda.Stream(device=dev)   # a capture needs a stream of its own
        with torch.cuda.graph(graph, stream=capture):
            wl.step(capture)
        torch.cuda.synchronize()
        run_step = graph.replay
        for _ in range(max(3, args.warmup)):
            run_step()
        torch.cuda.synchronize()
        if cpsa.cpp_read_device_error(wl.err) != 0:
            raise SystemExit("device error flags set during graph warm-up")
    clocks = ClockSampler(gpu_uuid)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    enqueue_s = []
    if dist: dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_wall = time.perf_counter()
    for s in range(args.steps):
        flush.zero_()
        ev0[s].record(stream)
        te = time.perf_counter()
        run_step()
        enqueue_s.append(time.perf_counter() - te)
        ev1[s].record(stream)
        torch.cuda.synchronize()
    torch.cuda.synchronize()
    if dist: dist.barrier()
    t_end = time.perf_counter()
    wall = t_end - t_wall
    clocks.mark(t_wall, t_end)
    clk = clocks.stop()
    step_ms = [ev0[s].elapsed_time(ev1[s]) for s in range(args.steps)]
    total_ms = max_over_ranks(float(sum(step_ms)), dist, dev)
    flags = cpsa.cpp_read_device_error(wl.err)
    ms_per_step = total_ms / args.steps
    value = job_tflops(world, STEP_FLOPS, args.steps, total_ms)

    # end-to-end through host buffers: the same launch mode as the headline (the
    # whole host-buffer step, copies included, captured once and replayed), and
    # the stream-launch variant beside it
    h2d, d2h = wl.make_host()
    for _ in range(2):
        wl.step_e2e(stream)
    torch.cuda.synchronize()

    def time_e2e(fn, reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ms = []
        for _ in range(reps):
            flush.zero_()
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        return float(np.mean(ms))

    e2e_eager_ms = time_e2e(lambda: wl.step_e2e(stream), max(1, args.steps // 2))
    e2e_run = None
    if not args.eager:
        e2e_graph = torch.cuda.CUDAGraph()
        capture2 = torch.cuda.Stream(device=dev)
        with torch.cuda.graph(e2e_graph, stream=capture2):
            wl.step_e2e(capture2)
        torch.cuda.synchronize()
        for _ in range(2):
            e2e_graph.replay()
        torch.cuda.synchronize()
        e2e_run = e2e_graph.replay
    e2e_step_ms = e2e_eager_ms if e2e_run is None else time_e2e(e2e_run, max(1, args.steps // 2))
    e2e_step_ms = max_over_ranks(e2e_step_ms, dist, dev)
    e2e_val = job_tflops(world, STEP_FLOPS, 1, e2e_step_ms)

    # roofline of the dominant kernel (the tensor-core chunk kernel): separate steps
    # with events around every chunk-kernel launch (the headline steps carry none),
    # in the headline's launch mode (the marked step captured in a graph of its own,
    # the events becoming event nodes around each kernel) and as stream launches
    def marked_steps(run):
        kernel_ms = []
        for _ in range(5):
            flush.zero_()
            run()
            torch.cuda.synchronize()
            kernel_ms.append(wl.chunk_kernel_ms())
        return np.asarray(kernel_ms)                 # [steps, chunks]

    km_stream = marked_steps(lambda: wl.step(stream, with_marks=True))
    km = km_stream
    if not args.eager:
        marked_graph = torch.cuda.CUDAGraph()
        capture3 = torch.cuda.Stream(device=dev)
        with torch.cuda.graph(marked_graph, stream=capture3):
            wl.step(capture3, with_marks=True)
        torch.cuda.synchronize()
        marked_graph.replay()
        torch.cuda.synchronize()
        km = marked_steps(marked_graph.replay)
    peak_tf, peak_bw, peak_src = load_peaks()
    per_launch_ms = float(km.mean())
    per_launch_flops = STEP_FLOPS / N_CHUNKS
    achieved = per_launch_flops / (per_launch_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak_tf, "unit": "TFLOP/s",
                "frac": round(achieved / peak_tf, 4), "traffic": load_traffic(),
                "kernel": "chunk_attn_kernel<128,2,true> (one request per call: runs planned by the kernel itself)", "peak_source": f"{peak_src} bf16 dense (burst)",
                "per_launch_flops": per_launch_flops, "per_launch_ms": round(per_launch_ms, 4),
                "launch": "stream launches" if args.eager else "graph replay (event nodes around each launch)",
                "per_launch_ms_stream_launches": round(float(km_stream.mean()), 4),
                "last_chunk_ms": round(float(km[:, -1].mean()), 4),
                "per_chunk_ms": [round(float(x), 4) for x in km.mean(axis=0)],
                "last_chunk_tflops": round(chunk_flops((N_CHUNKS - 1) * CHUNK, CHUNK) / (km[:, -1].mean() * 1e-3) / 1e12, 2)}
    # per chunk: split, [KV write,] chunk attention (a single prefill request of
    # 512 tokens plans its runs inside the chunk kernel and launches neither the
    # decode nor the combine kernel)
    launches = args.steps * N_CHUNKS * (2 if wl.fused else 3)

    # the same step as stream launches, beside the graph replays
    eager = {}
    if rank == 0 and not args.eager and not args.no_compare:
        ems = []
        o0, o1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(10):
            flush.zero_()
            o0.record(stream)
            eager_step()
            o1.record(stream)
            torch.cuda.synchronize()
            ems.append(o0.elapsed_time(o1))
        e_ms = float(np.mean(ems))
        eager = {"ms_per_step": round(e_ms, 4), "value": round(STEP_FLOPS / (e_ms * 1e-3) / 1e12, 3),
                 "device_flags": cpsa.cpp_read_device_error(wl.err)}

    # the other variant of the step (two calls, or the fused call) on the same inputs
    other = {}
    if rank == 0 and not args.no_compare:
        wl.fused = not wl.fused
        for _ in range(3):
            wl.step(stream)
        torch.cuda.synchronize()
        oms = []
        o0, o1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(10):
            flush.zero_()
            o0.record(stream)
            wl.step(stream)
            o1.record(stream)
            torch.cuda.synchronize()
            oms.append(o0.elapsed_time(o1))
        o_ms = float(np.mean(oms))
        other = {"ms_per_step": round(o_ms, 4), "value": round(STEP_FLOPS / (o_ms * 1e-3) / 1e12, 3),
                 "device_flags": cpsa.cpp_read_device_error(wl.err)}
        wl.fused = not wl.fused

    line = {"metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "ms_per_step_median": round(float(np.median(step_ms)), 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 q/k/v, permuted page pool)",
            "config": {"workload": WORKLOAD, "global_batch": world, "seq_len": SEQ, "chunk": CHUNK,
                       "kv_write": "fused into the attention call" if wl.fused else "separate call",
                       "launch": "stream launches" if args.eager else "one CUDA graph per step (replayed)",
                       "parallelism": "replicas" if world > 1 else "single-gpu",
                       "l2": "flushed between steps (256 MB write)", "max_kv_splits": wl.max_kv_splits,
                       "step_flops": STEP_FLOPS},
            "e2e": {"value": round(e2e_val, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_step_ms, 4),
                    "launch": "stream launches" if args.eager else "one CUDA graph per step (copies included)",
                    "stream_launch_ms_per_step": round(e2e_eager_ms, 4)},
            "roofline": roofline, "gpu_launches": launches, "clocks": clk,
            "tokens_per_s": round(world * SEQ / (ms_per_step * 1e-3), 1),
            "step_roofline": step_roofline(ms_per_step, peak_tf, peak_bw),
            "wall_s": round(wall, 3), "host_enqueue_ms_per_step": round(1e3 * float(np.mean(enqueue_s)), 3),
            "device_flags": flags}
    if eager:
        line["eager_step"] = eager
    if other:
        line["fused_step" if not wl.fused else "two_call_step"] = other
    if not args.no_secondary and rank == 0:
        del wl
        torch.cuda.empty_cache()
        try:
            line["kv_write"] = kv_write_bandwidth(dev)
            line["kv_write"]["hbm_peak_gbs"] = peak_bw
            line["kv_write"]["nominal_hbm_gbs"] = 8000.0
        except Exception as e:
            line["kv_write"] = {"error": repr(e)}
        try:
            line["secondary"] = decode_bandwidth(dev)
            line["secondary"]["hbm_peak_gbs"] = peak_bw
            line["secondary"]["decode_frac_of_hbm"] = round(line["secondary"]["decode_hbm_gbs"] / peak_bw, 4)
            # the same against the nominal HBM3e bandwidth the workload statement cites (about 8 TB/s)
            line["secondary"]["decode_frac_of_nominal_8tbs"] = round(line["secondary"]["decode_hbm_gbs"] / 8000.0, 4)
        except Exception as e:  # keep the headline line even if the secondary run fails
            line["secondary"] = {"error": repr(e)}
    if not args.no_suite and not args.no_secondary and rank == 0:
        try:
            line["suite"] = suite(dev)
        except Exception as e:
            line["suite"] = {"error": repr(e)}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(host_inputs())
    # the decode and KV-write bandwidths and a compact summary close the line, so
    # that a reader who keeps only its tail still has them
    for key in ("kv_write", "secondary"):
        if key in line:
            line[key] = line.pop(key)
    if rank == 0 and not args.no_secondary:
        line["summary"] = summary_of(line)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def summary_of(line):
    """The secondary figures in a few keys: decode and KV-write HBM GB/s against the
    measured copy bandwidth, the page-16 chunk and the micro-batch workload."""
    out = {}
    sec, kvw, su = line.get("secondary", {}), line.get("kv_write", {}), line.get("suite", {})
    if "decode_hbm_gbs" in sec:
        out["decode_hbm_gbs"] = round(sec["decode_hbm_gbs"], 1)
        out["decode_frac_of_measured_hbm"] = sec.get("decode_frac_of_hbm")
        out["decode_frac_of_nominal_8tbs"] = sec.get("decode_frac_of_nominal_8tbs")
        out["sarathi_chunk_page16_ms"] = round(sec.get("chunk_kernel_ms", float("nan")), 4)
        out["sarathi_chunk_page16_tflops"] = round(sec.get("chunk_tflops", float("nan")), 1)
    for k, v in kvw.items():
        if isinstance(v, dict) and "gbs" in v:
            out[f"kv_write_{k}_gbs"] = v["gbs"]
    mb = su.get("microbatch_two_streams", {})
    if "two_vs_one" in mb:
        out["microbatch_two_vs_one"] = round(mb["two_vs_one"], 4)
        out["microbatch_prefill_tflops_one_stream"] = round(mb["prefill_tflops_one_stream"], 1)
        out["microbatch_prefill_tflops_one_stream_fused_kv_write"] = round(
            mb["fused_kv_write"]["prefill_tflops_one_stream"], 1)
    sl = su.get("serving_loop", {}).get("budget_only", {})
    if "graph_replay_ms" in sl:
        out["serving_loop_ms_per_call_events"] = sl["device_ms"]
        out["serving_loop_ms_graph_replay"] = sl["graph_replay_ms"]
    if "tile_alignment_h8192" in su:
        out["tile_alignment_h8192_ms"] = su["tile_alignment_h8192"]
    out["headline_tflops"] = line.get("value")
    out["headline_launch"] = line.get("config", {}).get("launch")
    if "eager_step" in line:
        out["eager_step_tflops"] = line["eager_step"]["value"]
    out["roofline_frac"] = line.get("roofline", {}).get("frac")
    return out


def reference_arm(args, world, rank):
    """The oracle (fp64, host cores) timed on the same workload and metric."""
    if rank != 0:
        return
    import torch
    import oracle
    oracle.build()
    inputs = host_inputs()
    q, k, v, slots, bt = inputs
    rng = np.random.default_rng(1)
    # size one step's sample to ~2 s of CPU work
    s1, f1, _ = oracle_sample(q, k, v, slots, bt, 1, rng, chunks=[N_CHUNKS - 1])
    rows = int(max(1, min(CHUNK, 2.0 / (s1 / f1 * STEP_FLOPS / SEQ * N_CHUNKS))))
    for _ in range(args.warmup):
        oracle_sample(q, k, v, slots, bt, 1, rng, chunks=[0])
    tot_s, tot_f, tot_n = 0.0, 0.0, 0
    for _ in range(args.steps):
        s, f, n = oracle_sample(q, k, v, slots, bt, rows, rng)
        tot_s += s
        tot_f += f
        tot_n += n
    val = tot_f / tot_s / 1e12
    sample = f"{rows} query rows per chunk x 64 chunks per step (all 32 heads); {tot_n} rows, {tot_f / 1e9:.1f} GFLOP"
    print(json.dumps({"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": world,
                      "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_s * 1e3 / args.steps,
                      "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                      "data": "synthetic", "config": {"workload": WORKLOAD, "seq_len": SEQ, "chunk": CHUNK},
                      "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                                       "kind": "oracle", "sample": sample},
                      "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
          flush=True)
    del torch


if __name__ == "__main__":
    main()
