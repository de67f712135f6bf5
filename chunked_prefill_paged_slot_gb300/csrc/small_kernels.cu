// small_kernels.cu -- the KV write, the split-KV combine and the micro-batch split.
#include "common.cuh"
#include "kernels.cuh"
#include "plan.cuh"

namespace cpsa {

namespace {

// ---------------------------------------------------------------------------
// KV write ("Ascend dual-stream parallel" article, section 3.1, slot_mapping:
// every new token goes to its own cache slot). A bit copy in 16-byte vectors:
// thread x of a (token, kv head) row moves bytes [16x, 16x+16) of k and of v.
// Consecutive threads read consecutive bytes of k/v and write consecutive bytes
// of one cache row, so both sides are coalesced.
// ---------------------------------------------------------------------------
template <int VEC_PER_ROW>
__global__ void __launch_bounds__(256) kv_write_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                                       const int64_t *__restrict__ slot_mapping, int64_t num_tokens,
                                                       int num_kv_heads, int page_size, int64_t num_pages,
                                                       uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                                                       uint32_t *dev_err)
{
    pdl_trigger();
    pdl_wait();
    const int64_t rows = num_tokens * num_kv_heads;
    const int64_t total = rows * VEC_PER_ROW;
    const int64_t slots = num_pages * page_size;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / VEC_PER_ROW;
        const int x = (int)(i % VEC_PER_ROW);
        const int64_t t = row / num_kv_heads;
        const int h = (int)(row % num_kv_heads);
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0)
            continue;   // padding token
        if (slot >= slots) {
            if (h == 0 && x == 0)
                set_dev_error(dev_err, CPSA_DEV_SLOT_OUT_OF_RANGE);
            continue;
        }
        const int64_t page = slot / page_size;
        const int64_t off = slot - page * page_size;
        const int64_t dst = ((page * num_kv_heads + h) * page_size + off) * VEC_PER_ROW + x;
        const uint4 kv = __ldcs(k + i);
        const uint4 vv = __ldcs(v + i);
        k_cache[dst] = kv;
        v_cache[dst] = vv;
    }
}

// ---------------------------------------------------------------------------
// Combine of split rows: O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s,
// M = max_s m_s (m in base-2 units). Persistent: the (row, q head) units of all
// combine items are numbered consecutively (CombineItem::u0; an item covers
// nrows rows x nh heads from h0). Each CTA stages the items (all of them when
// they fit, else their first units) in shared memory; each warp takes two
// consecutive units at a time, lane l owning output columns [4l, 4l+4)
// (D = 128) or [2l, 2l+2) (D = 64). Both units' (m, l) and first partial O
// loads are in flight before any weight is formed: the kernel is bound by the
// latency of those loads, not by bandwidth.
// ---------------------------------------------------------------------------
constexpr int kCombineThreads = 256;
constexpr int kCombineSmemItems = 4096;    // first units staged for up to this many items
constexpr int kCombineFullItems = 512;     // whole items staged for up to this many
constexpr int kCombineMaxSplits = 32;
constexpr int kCombineRound = 4;           // partial O rows loaded per unit per round
constexpr int kCombineUnits = 2;           // units per warp in flight

template <int D>
__global__ void __launch_bounds__(kCombineThreads, 4) combine_kernel(const CombineParams p)
{
    __shared__ int s_u0[kCombineSmemItems];
    __shared__ CombineItem s_item[kCombineFullItems];
    pdl_trigger();
    pdl_wait();
    const int n_items = p.counts[kCntCombine];
    const int total = p.counts[kCntCombineUnits];
    if (n_items == 0 || total == 0)
        return;
    const bool staged = n_items <= kCombineSmemItems;
    const bool full = n_items <= kCombineFullItems;
    if (full) {
        for (int i = threadIdx.x; i < n_items; i += kCombineThreads) {
            s_item[i] = p.citems[i];
            s_u0[i] = s_item[i].u0;
        }
    } else if (staged) {
        for (int i = threadIdx.x; i < n_items; i += kCombineThreads) s_u0[i] = p.citems[i].u0;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (kCombineThreads / 32);
    constexpr int PER_LANE = D / 32;
    const int Hq = p.num_q_heads;
    auto find = [&](int u) -> CombineItem {   // the last item with u0 <= u
        int lo = 0, hi = n_items - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            const int v = staged ? s_u0[mid] : p.citems[mid].u0;
            if (v <= u) lo = mid; else hi = mid - 1;
        }
        return full ? s_item[lo] : p.citems[lo];
    };
    auto load_o = [&](float (&dst)[PER_LANE], int64_t row) {
        const float *src = p.part_o + row * D + lane * PER_LANE;
        if (PER_LANE == 4) {
            const float4 x = __ldcs(reinterpret_cast<const float4 *>(src));
            dst[0] = x.x; dst[1 % PER_LANE] = x.y; dst[2 % PER_LANE] = x.z; dst[3 % PER_LANE] = x.w;
        } else {
            const float2 x = __ldcs(reinterpret_cast<const float2 *>(src));
            dst[0] = x.x; dst[1 % PER_LANE] = x.y;
        }
    };
    constexpr int NU = kCombineUnits;
    for (int ub = (blockIdx.x * (kCombineThreads / 32) + (threadIdx.x >> 5)) * NU; ub < total; ub += warps * NU) {
        int64_t pr0[NU];   // first partial row of the unit
        int trow[NU], head[NU], ns[NU];
        bool live[NU];
        float2 ml[NU];
        float o[NU][kCombineRound][PER_LANE];
#pragma unroll
        for (int k = 0; k < NU; ++k) {
            live[k] = ub + k < total;
            pr0[k] = 0;
            trow[k] = head[k] = ns[k] = 0;
            if (live[k]) {
                const CombineItem c = find(ub + k);
                const int local = ub + k - c.u0;
                pr0[k] = (int64_t)c.pbase + (int64_t)local * c.nsplit;
                trow[k] = c.t0 + local / c.nh;
                head[k] = c.h0 + local % c.nh;
                ns[k] = c.nsplit;
            }
        }
        // every load of the first round, for all units, before any arithmetic
#pragma unroll
        for (int k = 0; k < NU; ++k) {
            ml[k] = lane < ns[k] ? __ldcs(reinterpret_cast<const float2 *>(p.part_ml) + pr0[k] + lane)
                                 : make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int j = 0; j < kCombineRound; ++j)
                if (j < ns[k])
                    load_o(o[k][j], pr0[k] + j);
        }
#pragma unroll
        for (int k = 0; k < NU; ++k) {
            if (!live[k])
                continue;
            float M = ml[k].x;
            for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
            const float Mref = M == -INFINITY ? 0.f : M;
            const float f = ex2_approx(ml[k].x - Mref);   // lane s: weight of split s
            float L = f * ml[k].y;
            for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
            float acc[PER_LANE];
#pragma unroll
            for (int e = 0; e < PER_LANE; ++e) acc[e] = 0.f;
#pragma unroll
            for (int j = 0; j < kCombineRound; ++j) {
                if (j < ns[k]) {
                    const float fs = __shfl_sync(0xffffffffu, f, j);
#pragma unroll
                    for (int e = 0; e < PER_LANE; ++e) acc[e] += fs * o[k][j][e];
                }
            }
            // more splits than one round (long decode rows): further rounds
            for (int s0 = kCombineRound; s0 < ns[k]; s0 += kCombineRound) {
#pragma unroll
                for (int j = 0; j < kCombineRound; ++j)
                    if (s0 + j < ns[k])
                        load_o(o[k][j], pr0[k] + s0 + j);
#pragma unroll
                for (int j = 0; j < kCombineRound; ++j) {
                    if (s0 + j < ns[k]) {
                        const float fs = __shfl_sync(0xffffffffu, f, s0 + j);
#pragma unroll
                        for (int e = 0; e < PER_LANE; ++e) acc[e] += fs * o[k][j][e];
                    }
                }
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
            __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.out) +
                                 ((int64_t)trow[k] * Hq + head[k]) * D + lane * PER_LANE;
#pragma unroll
            for (int e = 0; e < PER_LANE; e += 2)
                *reinterpret_cast<uint32_t *>(dst + e) = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
        }
    }
}

// ---------------------------------------------------------------------------
// Balanced micro-batch split ("Ascend dual-stream parallel" article, section
// 3.1, advanced method): nearest request boundary to total/2 over cumulative
// query_lens, smallest k on ties, then the balance and length thresholds.
// One CTA: a chunked block scan gives every boundary's cumulative count, and a
// lexicographic (distance, k) minimum picks the boundary.
// ---------------------------------------------------------------------------
constexpr int kSplitThreads = 1024;

__global__ void __launch_bounds__(kSplitThreads, 1)
split_kernel(const int32_t *__restrict__ query_lens, int num_reqs, float balance_threshold,
             int32_t length_threshold, int32_t *out3)
{
    __shared__ long long warp_tot[kSplitThreads / 32];
    __shared__ unsigned long long warp_best[kSplitThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    pdl_trigger();
    pdl_wait();
    if (num_reqs < 2) {
        if (threadIdx.x == 0) {
            out3[0] = 0;
            out3[1] = 0;
            out3[2] = 0;
        }
        return;
    }
    // total
    long long tot = 0;
    for (int r = threadIdx.x; r < num_reqs; r += kSplitThreads) tot += query_lens[r];
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    if (lane == 0) warp_tot[warp] = tot;
    __syncthreads();
    long long total = 0;
    for (int w = 0; w < kSplitThreads / 32; ++w) total += warp_tot[w];
    __syncthreads();
    const long long best = total / 2;
    // cum_k = sum of query_lens[0 .. k-1] for k = 1 .. num_reqs-1, i.e. the
    // inclusive prefix at r = k-1; key = (|cum_k - best| << 24 | k) -- k < 2^24
    unsigned long long my_best = ~0ull;
    long long carry = 0;
    for (int base = 0; base < num_reqs - 1; base += kSplitThreads) {
        const int r = base + threadIdx.x;
        long long x = r < num_reqs - 1 ? query_lens[r] : 0;
        for (int o = 1; o < 32; o <<= 1) {
            long long y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        long long before = 0, chunk = 0;
        for (int w = 0; w < kSplitThreads / 32; ++w) {
            if (w < warp) before += warp_tot[w];
            chunk += warp_tot[w];
        }
        __syncthreads();
        if (r < num_reqs - 1) {
            const long long cum = carry + before + x;
            const long long diff = cum > best ? cum - best : best - cum;
            const unsigned long long key = ((unsigned long long)diff << 24) | (unsigned long long)(r + 1);
            if (key < my_best) my_best = key;
        }
        carry += chunk;
    }
    for (int o = 16; o > 0; o >>= 1) {
        unsigned long long y = __shfl_xor_sync(0xffffffffu, my_best, o);
        if (y < my_best) my_best = y;
    }
    if (lane == 0) warp_best[warp] = my_best;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long b = ~0ull;
        for (int w = 0; w < kSplitThreads / 32; ++w)
            if (warp_best[w] < b) b = warp_best[w];
        const int k = (int)(b & 0xFFFFFFull);
        long long n1 = 0;
        for (int r = 0; r < k; ++r) n1 += query_lens[r];
        const long long n2 = total - n1;
        const long long small = n1 < n2 ? n1 : n2;
        int use_two = 0;
        if (small > 0) {
            const long long gap = n1 > n2 ? n1 - n2 : n2 - n1;
            const bool balanced = (double)gap / (double)small <= (double)balance_threshold;
            use_two = balanced && small >= (long long)length_threshold;
        }
        out3[0] = k;
        out3[1] = (int32_t)n1;
        out3[2] = use_two;
    }
}

// Both exp2 paths of the attention kernels on an array: the FMA-pipe polynomial
// (inputs clamped to [-125, 127] as the kernels do) and the hardware ex2.approx.
__global__ void exp2_selftest_kernel(const float *x, float *poly, float *hw, int64_t n)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float v = x[i];
        const float c = fminf(fmaxf(v, -125.0f), 127.0f);
        float lo, hi;
        f2_unpack(exp2_poly_x2(f2_pack(c, c)), lo, hi);
        poly[i] = lo;
        hw[i] = ex2_approx(v);
    }
}

// Self-test of the bounded waits every kernel of the path uses (mbar_wait,
// mbar_wait_sleep) and of the abort hand-off between a CTA's roles. Warp 0
// waits, busy-polling, on an mbarrier that nothing arrives at, with the limit
// the caller passes; when it runs out it sets the CTA's abort flag. Warp 1
// waits, sleeping between polls, on a second such barrier with the kernels'
// standard limit (one second): it must leave as soon as it sees the abort flag,
// long before its own limit. Thread 0 then raises CPSA_DEV_WAIT_TIMEOUT exactly
// as the attention kernels do. out[0], out[1]: whether each wait succeeded (1)
// or gave up (0); out[2]: microseconds warp 1 waited. No copy or MMA is in
// flight at any point, so the CTA ends as soon as both waits return.
__global__ void wait_selftest_kernel(uint64_t limit_ns, uint32_t *dev_err, int32_t *out)
{
    __shared__ __align__(8) uint64_t bar_a, bar_b;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar_a, 1);
        mbar_init(&bar_b, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    volatile int *abort = &abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        const bool ok = mbar_wait(&bar_a, 0, abort, limit_ns);
        if (lane == 0)
            out[0] = ok ? 1 : 0;
    } else if (warp == 1) {
        const uint64_t t0 = global_timer_ns();
        const bool ok = mbar_wait_sleep(&bar_b, 0, abort);
        const uint64_t us = (global_timer_ns() - t0) / 1000u;
        if (lane == 0) {
            out[1] = ok ? 1 : 0;
            out[2] = (int32_t)(us < 0x7fffffffu ? us : 0x7fffffffu);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort)
        set_dev_error(dev_err, CPSA_DEV_WAIT_TIMEOUT);
}

// The same split for batches of at most kSplitSmallMax requests, by one warp
// with no shared memory: the running prefix is carried across 32-request
// chunks, and the winning boundary carries its own prefix, so n1 needs no second
// pass. A lone warp fits beside a chunk-kernel CTA on its SM, so it can start
// as soon as the attention call before it ends.
constexpr int kSplitSmallMax = 256;

__global__ void __launch_bounds__(32, 1)
split_small_kernel(const int32_t *__restrict__ query_lens, int num_reqs, float balance_threshold,
                   int32_t length_threshold, int32_t *out3)
{
    const int lane = threadIdx.x;
    pdl_trigger();
    pdl_wait();
    if (num_reqs < 2) {
        if (lane == 0) {
            out3[0] = 0;
            out3[1] = 0;
            out3[2] = 0;
        }
        return;
    }
    long long total = 0;
    for (int r = lane; r < num_reqs; r += 32) total += query_lens[r];
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    const long long best = total / 2;
    // key = (|cum_k - best| << 24 | k) for k = 1 .. num_reqs-1 (cum_k: inclusive prefix at r = k-1)
    unsigned long long my_best = ~0ull;
    long long my_cum = 0, carry = 0;
    for (int base = 0; base < num_reqs - 1; base += 32) {
        const int r = base + lane;
        long long x = r < num_reqs - 1 ? query_lens[r] : 0;
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (r < num_reqs - 1) {
            const long long cum = carry + x;
            const long long diff = cum > best ? cum - best : best - cum;
            const unsigned long long key = ((unsigned long long)diff << 24) | (unsigned long long)(r + 1);
            if (key < my_best) {
                my_best = key;
                my_cum = cum;
            }
        }
        carry += __shfl_sync(0xffffffffu, x, 31);
    }
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, my_best, o);
        const long long c = __shfl_xor_sync(0xffffffffu, my_cum, o);
        if (y < my_best) {
            my_best = y;
            my_cum = c;
        }
    }
    if (lane == 0) {
        const int k = (int)(my_best & 0xFFFFFFull);
        const long long n1 = my_cum;
        const long long n2 = total - n1;
        const long long small = n1 < n2 ? n1 : n2;
        int use_two = 0;
        if (small > 0) {
            const long long gap = n1 > n2 ? n1 - n2 : n2 - n1;
            const bool balanced = (double)gap / (double)small <= (double)balance_threshold;
            use_two = balanced && small >= (long long)length_threshold;
        }
        out3[0] = k;
        out3[1] = (int32_t)n1;
        out3[2] = use_two;
    }
}

}  // namespace

cudaError_t launch_exp2_selftest(const float *x, float *poly, float *hw, int64_t n, cudaStream_t s)
{
    if (n <= 0)
        return cudaSuccess;
    exp2_selftest_kernel<<<(int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024), 256, 0, s>>>(x, poly, hw, n);
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, uint32_t *dev_err, int32_t *out, cudaStream_t s)
{
    wait_selftest_kernel<<<1, 64, 0, s>>>(limit_ns, dev_err, out);
    return cudaGetLastError();
}

cudaError_t launch_kv_cache_write(const void *k, const void *v, const int64_t *slot_mapping, int64_t num_tokens,
                                  int num_kv_heads, int head_dim, int page_size, int64_t num_pages, void *k_cache,
                                  void *v_cache, uint32_t *dev_err, int num_sms, cudaStream_t s)
{
    const int64_t total = num_tokens * num_kv_heads * (head_dim / 8);
    if (total == 0)
        return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (head_dim == 128)
        return launch_pdl(false, kv_write_kernel<16>, dim3((unsigned)blocks), dim3(256), 0, s, (const uint4 *)k,
                          (const uint4 *)v, slot_mapping, num_tokens, num_kv_heads, page_size, num_pages,
                          (uint4 *)k_cache, (uint4 *)v_cache, dev_err);
    return launch_pdl(false, kv_write_kernel<8>, dim3((unsigned)blocks), dim3(256), 0, s, (const uint4 *)k,
                      (const uint4 *)v, slot_mapping, num_tokens, num_kv_heads, page_size, num_pages,
                      (uint4 *)k_cache, (uint4 *)v_cache, dev_err);
}

cudaError_t launch_combine(const CombineParams &p, int head_dim, int grid, cudaStream_t s, bool early)
{
    if (head_dim == 128)
        return launch_pdl(early, combine_kernel<128>, dim3(grid), dim3(kCombineThreads), 0, s, p);
    return launch_pdl(early, combine_kernel<64>, dim3(grid), dim3(kCombineThreads), 0, s, p);
}

cudaError_t launch_split_microbatch(const int32_t *query_lens, int num_reqs, float balance_threshold,
                                    int32_t length_threshold, int32_t *out3, cudaStream_t s)
{
    if (num_reqs <= kSplitSmallMax)
        return launch_pdl(false, split_small_kernel, dim3(1), dim3(32), 0, s, query_lens, num_reqs, balance_threshold,
                          length_threshold, out3);
    return launch_pdl(false, split_kernel, dim3(1), dim3(kSplitThreads), 0, s, query_lens, num_reqs, balance_threshold,
                      length_threshold, out3);
}

}  // namespace cpsa
