// plan.cu -- the metadata step of one attention call, as a single-CTA kernel.
//
// From query_lens / seq_lens ("Ascend dual-stream parallel" article, section 3.1:
// seq_lens = history plus current tokens, query_lens = current tokens) it builds
//   cu_q      exclusive scan of query_lens (row offset of every request in q/out),
//   checks    seq_len >= query_len >= 0, seq_len fits the block_table row, and
//             sum(query_lens) == num_tokens,
//   items     prefill items (query tile x kv head x head pair x KV split), decode
//             items (row x kv head x KV split) and combine items,
// and stores the counts that the persistent kernels read.
// Two passes over the requests: the first sums the partial rows needed, so that
// when they exceed the workspace every row falls back to one split; the second
// scans and writes the lists.
#include "common.cuh"
#include "plan.cuh"

namespace cpsa {

namespace {

constexpr int kPlanThreads = 1024;

struct ReqCounts {
    int q;        // query_len used in the row scan (0 when the request is invalid)
    int pitems;
    int ditems;
    int citems;
    int prows;
    int cunits;   // (row, q head) units to combine
};
constexpr int kScan = 6;

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Per-request work: counts (emit == false) or the lists themselves (emit == true).
__device__ void request_work(const PlanParams &p, int r, int max_splits, bool emit, int q_off,
                             int pitem_off, int ditem_off, int citem_off, int prow_off, int cunit_off,
                             ReqCounts &c)
{
    c = ReqCounts{0, 0, 0, 0, 0, 0};
    int q = p.query_lens[r];
    int s = p.seq_lens[r];
    bool valid = true;
    if (q < 0 || s < q) {
        if (emit) set_dev_error(p.dev_err, CPSA_DEV_SEQ_LT_QUERY);
        valid = false;
    } else if ((int64_t)s > (int64_t)p.max_blocks * p.page_size) {
        if (emit) set_dev_error(p.dev_err, CPSA_DEV_SEQ_GT_TABLE);
        valid = false;
    }
    c.q = q > 0 ? q : 0;   // invalid requests still occupy their rows in q / out
    if (!valid || q == 0)
        return;
    int hist = s - q;
    if (q == 1) {
        // decode row: splits along keys, in whole pipeline stages
        int nch = ceil_div(s, kDecodeChunk);
        int ns = ceil_div(s, kDecodeKeysPerSplit);
        if (ns > max_splits) ns = max_splits;
        if (ns > nch) ns = nch;
        if (ns < 1) ns = 1;
        c.ditems = p.Hkv * ns;
        if (ns > 1) {
            c.prows = p.Hq * ns;
            c.citems = 1;
            c.cunits = p.Hq;
        }
        if (emit) {
            int k = 0;
            for (int sp = 0; sp < ns; ++sp) {
                const int c0 = sp * nch / ns, c1 = (sp + 1) * nch / ns;
                const int key1 = min(c1 * kDecodeChunk, s);
                for (int kvh = 0; kvh < p.Hkv; ++kvh)
                    p.ditems[ditem_off + k++] = DecodeItem{r, kvh, c0 * kDecodeChunk, key1, sp, ns,
                                                           ns > 1 ? prow_off : -1, q_off};
            }
            if (ns > 1)
                p.citems[citem_off] = CombineItem{q_off, 1, prow_off, ns, cunit_off, 0, 0, 0};
        }
        return;
    }
    // prefill: 128-row query tiles, longest KV range first
    int nqt = ceil_div(q, kTileM);
    int pairs = p.group / p.nq;
    int pi = 0, ci = 0, pr = 0, cu = 0;
    for (int qt = nqt - 1; qt >= 0; --qt) {
        const int i0 = qt * kTileM;
        const int rows = q - i0 < kTileM ? q - i0 : kTileM;
        const int nkv = ceil_div(hist + i0 + rows, kTileN);
        int ns = ceil_div(nkv, kPrefillTilesPerSplit);
        if (ns > max_splits) ns = max_splits;
        if (ns < 1) ns = 1;
        const int pbase = ns > 1 ? prow_off + pr : -1;
        if (emit) {
            // splits outermost: items of one split sit together and cover all heads
            for (int sp = 0; sp < ns; ++sp) {
                const int kt0 = sp * nkv / ns, kt1 = (sp + 1) * nkv / ns;
                for (int kvh = 0; kvh < p.Hkv; ++kvh)
                    for (int hp = 0; hp < pairs; ++hp)
                        p.pitems[pitem_off + pi++] = PrefillItem{r, i0, kvh | (hp << 16), kt0, kt1, sp, ns, pbase};
            }
            if (ns > 1)
                p.citems[citem_off + ci] = CombineItem{q_off + i0, rows, pbase, ns, cunit_off + cu, 0, 0, 0};
        } else {
            pi += p.Hkv * pairs * ns;
        }
        if (ns > 1) {
            pr += rows * p.Hq * ns;
            cu += rows * p.Hq;
            ++ci;
        }
    }
    c.pitems = pi;
    c.citems = ci;
    c.prows = pr;
    c.cunits = cu;
}

// Block-wide exclusive scan of kScan ints (kPlanThreads threads); returns the totals.
__device__ void block_scan(int (&v)[kScan], int (&tot)[kScan])
{
    __shared__ int warp_sums[kPlanThreads / 32][kScan];
    int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl[kScan];
#pragma unroll
    for (int j = 0; j < kScan; ++j) {
        int x = v[j];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        incl[j] = x;
    }
    if (lane == 31)
        for (int j = 0; j < kScan; ++j) warp_sums[warp][j] = incl[j];
    __syncthreads();
    if (warp == 0) {
        for (int j = 0; j < kScan; ++j) {
            int x = warp_sums[lane][j];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            warp_sums[lane][j] = x;   // inclusive over warps
        }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kScan; ++j) {
        int before = warp > 0 ? warp_sums[warp - 1][j] : 0;
        tot[j] = warp_sums[kPlanThreads / 32 - 1][j];
        v[j] = before + incl[j] - v[j];
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(PlanParams p)
{
    __shared__ int s_clamp;
    // pass 1: totals
    int64_t tok = 0, prows = 0;
    for (int base = 0; base < p.num_reqs; base += kPlanThreads) {
        int r = base + threadIdx.x;
        ReqCounts c{0, 0, 0, 0, 0, 0};
        if (r < p.num_reqs)
            request_work(p, r, p.max_splits, false, 0, 0, 0, 0, 0, 0, c);
        tok += c.q;
        prows += c.prows;
    }
    // reduce tok and prows over the block
    __shared__ long long red[2][kPlanThreads / 32];
    long long a = tok, b = prows;
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
    }
    if ((threadIdx.x & 31) == 0) {
        red[0][threadIdx.x >> 5] = a;
        red[1][threadIdx.x >> 5] = b;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        long long ta = 0, tb = 0;
        for (int w = 0; w < kPlanThreads / 32; ++w) {
            ta += red[0][w];
            tb += red[1][w];
        }
        int clamp = 0;
        if (ta != p.num_tokens) {
            set_dev_error(p.dev_err, CPSA_DEV_TOKENS_MISMATCH);
            clamp = 2;
        } else if (tb > p.prow_capacity) {
            set_dev_error(p.dev_err, CPSA_DEV_SPLITS_CLAMPED);
            clamp = 1;
        }
        s_clamp = clamp;
    }
    __syncthreads();
    if (s_clamp == 2) {
        if (threadIdx.x < kCntSlots) p.counts[threadIdx.x] = 0;
        return;
    }
    int max_splits = s_clamp ? 1 : p.max_splits;
    // pass 2: scans and lists
    int carry[kScan] = {0, 0, 0, 0, 0, 0};
    for (int base = 0; base < p.num_reqs; base += kPlanThreads) {
        int r = base + threadIdx.x;
        ReqCounts c{0, 0, 0, 0, 0, 0};
        if (r < p.num_reqs)
            request_work(p, r, max_splits, false, 0, 0, 0, 0, 0, 0, c);
        int v[kScan] = {c.q, c.pitems, c.ditems, c.citems, c.prows, c.cunits};
        int tot[kScan];
        block_scan(v, tot);
        if (r < p.num_reqs) {
            p.cu_q[r] = carry[0] + v[0];
            bool fits = carry[1] + v[1] + c.pitems <= p.max_pitems &&
                        carry[2] + v[2] + c.ditems <= p.max_ditems &&
                        carry[3] + v[3] + c.citems <= p.max_citems;
            if (fits)
                request_work(p, r, max_splits, true, carry[0] + v[0], carry[1] + v[1],
                             carry[2] + v[2], carry[3] + v[3], carry[4] + v[4], carry[5] + v[5], c);
        }
        for (int j = 0; j < kScan; ++j) carry[j] += tot[j];
    }
    if (threadIdx.x == 0) {
        p.cu_q[p.num_reqs] = carry[0];
        p.counts[kCntPrefill] = carry[1] < p.max_pitems ? carry[1] : (int)p.max_pitems;
        p.counts[kCntDecode] = carry[2] < p.max_ditems ? carry[2] : (int)p.max_ditems;
        p.counts[kCntCombine] = carry[3] < p.max_citems ? carry[3] : (int)p.max_citems;
        p.counts[kCntPartialRows] = carry[4];
        p.counts[kCntCombineUnits] = carry[5];
        for (int j = 5; j < kCntSlots; ++j) p.counts[j] = 0;
    }
}

}  // namespace

void launch_plan(const PlanParams &p, cudaStream_t s)
{
    plan_kernel<<<1, kPlanThreads, 0, s>>>(p);
}

}  // namespace cpsa
