// plan.cu -- the metadata step of one attention call, as a single-CTA kernel.
//
// From query_lens / seq_lens ("Ascend dual-stream parallel" article, section 3.1:
// seq_lens = history plus current tokens, query_lens = current tokens) it builds
//   cu_q      exclusive scan of query_lens (row offset of every request in q/out),
//   checks    seq_len >= query_len >= 0, seq_len fits the block_table row, and
//             sum(query_lens) == num_tokens,
//   pieces    the stream-K cut of all prefill units' KV tiles into one run per
//             chunk-kernel CTA (see plan.cuh), decode items, combine items,
// and stores the counts that the persistent kernels read.
// Pass 1 sums tokens, prefill tiles (W) and decode partial rows, which fixes the
// run length and whether the partials fit the workspace (if not, nothing is
// split). Pass 2 walks the requests in chunks of 1024: one block scan gives each
// request its token and tile offsets, a second gives its list offsets, and each
// thread then writes its own request's entries.
#include "common.cuh"
#include "plan.cuh"

namespace cpsa {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kScan = 5;

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

struct Req {
    bool valid;
    int q, s, hist;
};

__device__ Req load_req(const PlanParams &p, int r)
{
    Req q;
    q.q = p.query_lens[r];
    q.s = p.seq_lens[r];
    q.valid = !(q.q < 0 || q.s < q.q) && (int64_t)q.s <= (int64_t)p.max_blocks * p.page_size;
    q.hist = q.s - q.q;
    return q;
}

// KV tiles of all prefill units of one request (0 for decode / invalid / empty).
__device__ int prefill_tiles(const PlanParams &p, const Req &rq)
{
    if (!rq.valid || rq.q < 2)
        return 0;
    const int units_per_qtile = p.Hkv * (p.group / p.nq);
    int tiles = 0;
    for (int i0 = 0; i0 < rq.q; i0 += kTileM) {
        const int rows = min(kTileM, rq.q - i0);
        tiles += ceil_div(rq.hist + i0 + rows, kTileN) * units_per_qtile;
    }
    return tiles;
}

__device__ int decode_splits(const Req &rq, int max_splits)
{
    const int nch = ceil_div(rq.s, kDecodeChunk);
    int ns = ceil_div(rq.s, kDecodeKeysPerSplit);
    ns = min(ns, max_splits);
    ns = min(ns, nch);
    return max(ns, 1);
}

// pieces; partial rows; combine units and combine items (split decode rows and
// split prefill units); decode items
struct Counts {
    int pieces, prows, cunits, citems, ditems;
};

__device__ __forceinline__ int warp_excl_scan(int x, int lane, int &total)
{
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    total = __shfl_sync(0xffffffffu, incl, 31);
    return incl - x;
}

// One request's work, walked by a whole warp (all arguments warp-uniform).
// With emit == false only the counts are returned (warp-uniform); with
// emit == true the entries are written at the given offsets, the lanes sharing
// the units of each query tile and placing them by warp scans.
// tile_off: global index of the request's first prefill tile; run: tiles per CTA
// run; cut: whether a run boundary may split a unit (else a unit goes whole to
// the run that holds its first tile).
__device__ Counts request_work(const PlanParams &p, int r, const Req &rq, int tile_off, int run, bool cut,
                               int max_splits, bool emit, int q_off, const Counts &off, int lane)
{
    Counts c{0, 0, 0, 0, 0};
    if (!rq.valid || rq.q == 0)
        return c;
    if (rq.q == 1) {
        const int ns = decode_splits(rq, max_splits);
        const int nch = ceil_div(rq.s, kDecodeChunk);
        c.ditems = p.Hkv * ns;
        if (ns > 1) {
            c.prows = p.Hq * ns;
            c.citems = 1;
            c.cunits = p.Hq;
        }
        if (emit) {
            for (int k = lane; k < c.ditems; k += 32) {
                const int sp = k / p.Hkv, kvh = k % p.Hkv;
                const int c0 = sp * nch / ns, c1 = (sp + 1) * nch / ns;
                const int key1 = min(c1 * kDecodeChunk, rq.s);
                p.ditems[off.ditems + k] = DecodeItem{r, kvh, c0 * kDecodeChunk, key1, sp, ns,
                                                      ns > 1 ? off.prows : -1, q_off};
            }
            if (ns > 1 && lane == 0)
                p.citems[off.citems] = CombineItem{q_off, 1, 0, p.Hq, off.prows, ns, off.cunits, 0};
        }
        return c;
    }
    // prefill units in order: query tiles (longest KV range first), kv heads, head pairs
    const int pairs = p.group / p.nq;
    const int upq = p.Hkv * pairs;            // units per query tile
    const int nqt = ceil_div(rq.q, kTileM);
    int tile_run = tile_off;
    for (int qt = nqt - 1; qt >= 0; --qt) {
        const int i0 = qt * kTileM;
        const int rows = min(kTileM, rq.q - i0);
        const int nkv = ceil_div(rq.hist + i0 + rows, kTileN);
        for (int jb = 0; jb < upq; jb += 32) {
            const int j = jb + lane;
            const bool active = j < upq;
            const int u0 = tile_run + j * nkv, u1 = u0 + nkv;
            const int np = active ? (cut ? (u1 - 1) / run - u0 / run + 1 : 1) : 0;
            const bool split = np > 1;
            int t_np, t_ci, t_pr, t_cu;
            const int e_np = warp_excl_scan(np, lane, t_np);
            const int e_ci = warp_excl_scan(split ? 1 : 0, lane, t_ci);
            const int e_pr = warp_excl_scan(split ? rows * p.nq * np : 0, lane, t_pr);
            const int e_cu = warp_excl_scan(split ? rows * p.nq : 0, lane, t_cu);
            if (emit && active) {
                const int kvh = j / pairs, hp = j % pairs;
                const int pbase = split ? off.prows + c.prows + e_pr : -1;
                const int pi = off.pieces + c.pieces + e_np;
                if (!split) {
                    p.pitems[pi] = PrefillItem{r, i0, kvh | (hp << 16), 0, nkv, (1 << 16), -1, u0 / run};
                } else {
                    int x = u0;
                    for (int pc = 0; pc < np; ++pc) {
                        const int owner = x / run;
                        const int end = min(u1, (owner + 1) * run);
                        p.pitems[pi + pc] =
                            PrefillItem{r, i0, kvh | (hp << 16), x - u0, end - u0, pc | (np << 16), pbase, owner};
                        x = end;
                    }
                    p.citems[off.citems + c.citems + e_ci] =
                        CombineItem{q_off + i0, rows, kvh * p.group + hp * p.nq, p.nq, pbase, np,
                                    off.cunits + c.cunits + e_cu, 0};
                }
            }
            c.pieces += t_np;
            c.citems += t_ci;
            c.prows += t_pr;
            c.cunits += t_cu;
        }
        tile_run += upq * nkv;
    }
    return c;
}

// Block-wide exclusive scan of N ints; returns the totals.
template <int N>
__device__ void block_scan(int (&v)[N], int (&tot)[N])
{
    __shared__ int warp_sums[kPlanThreads / 32][kScan];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl[N];
#pragma unroll
    for (int j = 0; j < N; ++j) {
        int x = v[j];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        incl[j] = x;
    }
    if (lane == 31)
        for (int j = 0; j < N; ++j) warp_sums[warp][j] = incl[j];
    __syncthreads();
    if (warp == 0) {
        for (int j = 0; j < N; ++j) {
            int x = warp_sums[lane][j];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            warp_sums[lane][j] = x;   // inclusive over warps
        }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < N; ++j) {
        const int before = warp > 0 ? warp_sums[warp - 1][j] : 0;
        tot[j] = warp_sums[kPlanThreads / 32 - 1][j];
        v[j] = before + incl[j] - v[j];
    }
    __syncthreads();
}

template <typename T>
__device__ T block_sum(T x)
{
    __shared__ long long red[kPlanThreads / 32];
    long long a = x;
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
    __syncthreads();
    long long t = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w) t += red[w];
    __syncthreads();
    return (T)t;
}

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(PlanParams p)
{
    // ---- pass 1: tokens, prefill tiles, decode partial rows
    long long tok = 0, tiles = 0, dprows = 0;
    for (int base = 0; base < p.num_reqs; base += kPlanThreads) {
        const int r = base + threadIdx.x;
        if (r < p.num_reqs) {
            const Req rq = load_req(p, r);
            tok += rq.q > 0 ? rq.q : 0;   // invalid requests still occupy their rows
            tiles += prefill_tiles(p, rq);
            if (rq.valid && rq.q == 1) {
                const int ns = decode_splits(rq, p.max_splits);
                if (ns > 1) dprows += (long long)p.Hq * ns;
            }
        }
    }
    tok = block_sum(tok);
    tiles = block_sum(tiles);
    dprows = block_sum(dprows);
    if (tok != p.num_tokens) {
        if (threadIdx.x == 0) set_dev_error(p.dev_err, CPSA_DEV_TOKENS_MISMATCH);
        if (threadIdx.x < kCntSlots) p.counts[threadIdx.x] = 0;
        for (int c = threadIdx.x; c <= p.chunk_grid; c += kPlanThreads) p.run_first[c] = 0;
        return;
    }
    // stream-K run length; cuts inside units only when splitting is allowed and
    // the partials' bound fits the workspace
    const int grid = max(1, p.chunk_grid);
    int run = (int)((tiles + grid - 1) / grid);
    run = max(run, kMinRunTiles);
    const long long pbound = (long long)2 * grid * kTileM * p.nq;
    int max_splits = p.max_splits;
    bool split_prefill = max_splits > 1;
    if (max_splits > 1 && pbound + dprows > p.prow_capacity) {
        if (threadIdx.x == 0) set_dev_error(p.dev_err, CPSA_DEV_SPLITS_CLAMPED);
        max_splits = 1;
        split_prefill = false;
    }

    // ---- pass 2: offsets and lists, 1024 requests at a time
    __shared__ int s_qoff[kPlanThreads], s_toff[kPlanThreads];
    __shared__ int s_cnt[kPlanThreads][kScan];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int carry_a[2] = {0, 0};                        // tokens, tiles
    int carry_b[kScan] = {0, 0, 0, 0, 0};           // pieces, prows, cunits, citems, ditems
    for (int base = 0; base < p.num_reqs; base += kPlanThreads) {
        const int nloc = min(kPlanThreads, p.num_reqs - base);
        // (a) token and tile offsets: one thread per request
        {
            const int r = base + threadIdx.x;
            int va[2] = {0, 0};
            if (threadIdx.x < nloc) {
                const Req rq = load_req(p, r);
                va[0] = rq.q > 0 ? rq.q : 0;
                va[1] = prefill_tiles(p, rq);
                if (!rq.valid)
                    set_dev_error(p.dev_err, (rq.q < 0 || rq.s < rq.q) ? CPSA_DEV_SEQ_LT_QUERY : CPSA_DEV_SEQ_GT_TABLE);
            }
            int ta[2];
            block_scan<2>(va, ta);
            s_qoff[threadIdx.x] = carry_a[0] + va[0];
            s_toff[threadIdx.x] = carry_a[1] + va[1];
            if (threadIdx.x < nloc)
                p.cu_q[r] = carry_a[0] + va[0];
            carry_a[0] += ta[0];
            carry_a[1] += ta[1];
        }
        __syncthreads();
        // (b) per-request counts: one warp per request
        for (int l = warp; l < nloc; l += kPlanThreads / 32) {
            const Req rq = load_req(p, base + l);
            const Counts c = request_work(p, base + l, rq, s_toff[l], run, split_prefill, max_splits, false,
                                          s_qoff[l], Counts{0, 0, 0, 0, 0}, lane);
            if (lane == 0) {
                s_cnt[l][0] = c.pieces;
                s_cnt[l][1] = c.prows;
                s_cnt[l][2] = c.cunits;
                s_cnt[l][3] = c.citems;
                s_cnt[l][4] = c.ditems;
            }
        }
        __syncthreads();
        // (c) list offsets: one thread per request
        {
            int vb[kScan];
            for (int j = 0; j < kScan; ++j) vb[j] = threadIdx.x < nloc ? s_cnt[threadIdx.x][j] : 0;
            int tb[kScan];
            block_scan<kScan>(vb, tb);   // ends with a barrier: s_cnt reads are done
            for (int j = 0; j < kScan; ++j) s_cnt[threadIdx.x][j] = carry_b[j] + vb[j];
            for (int j = 0; j < kScan; ++j) carry_b[j] += tb[j];
        }
        __syncthreads();
        // (d) the lists: one warp per request
        for (int l = warp; l < nloc; l += kPlanThreads / 32) {
            const Req rq = load_req(p, base + l);
            const Counts off{s_cnt[l][0], s_cnt[l][1], s_cnt[l][2], s_cnt[l][3], s_cnt[l][4]};
            request_work(p, base + l, rq, s_toff[l], run, split_prefill, max_splits, true, s_qoff[l], off, lane);
        }
        __syncthreads();
    }
    // run_first[c] = first piece whose owner is >= c (pieces are sorted by owner)
    __syncthreads();   // this block's piece writes are visible to the whole block
    const int n_pieces = (int)min((int64_t)carry_b[0], p.max_pitems);
    for (int i = threadIdx.x; i <= n_pieces; i += kPlanThreads) {
        const int lo = i == 0 ? 0 : p.pitems[i - 1].owner + 1;
        const int hi = i == n_pieces ? grid : p.pitems[i].owner;
        for (int c = lo; c <= hi; ++c) p.run_first[c] = i;
    }
    if (threadIdx.x == 0) {
        p.cu_q[p.num_reqs] = carry_a[0];
        p.counts[kCntPrefill] = (int)min((int64_t)carry_b[0], p.max_pitems);
        p.counts[kCntCombine] = (int)min((int64_t)carry_b[3], p.max_citems);
        p.counts[kCntPartialRows] = carry_b[1];
        p.counts[kCntCombineUnits] = carry_b[2];
        p.counts[kCntDecode] = (int)min((int64_t)carry_b[4], p.max_ditems);
        p.counts[kCntRunTiles] = run;
        for (int j = kCntRunTiles + 1; j < kCntSlots; ++j) p.counts[j] = 0;
    }
}

}  // namespace

void launch_plan(const PlanParams &p, cudaStream_t s)
{
    plan_kernel<<<1, kPlanThreads, 0, s>>>(p);
}

}  // namespace cpsa
