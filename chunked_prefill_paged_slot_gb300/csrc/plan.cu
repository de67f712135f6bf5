// plan.cu -- the metadata step of one attention call, as a single-CTA kernel.
//
// From query_lens / seq_lens ("Ascend dual-stream parallel" article, section 3.1:
// seq_lens = history plus current tokens, query_lens = current tokens) it builds
//   cu_q      exclusive scan of query_lens (row offset of every request in q/out),
//   checks    seq_len >= query_len >= 0, seq_len fits the block_table row, and
//             sum(query_lens) == num_tokens,
//   pieces    the stream-K cut of all prefill units' KV tiles into one run per
//             chunk-kernel CTA (see plan.cuh), decode items, combine items,
//             (the merge counters of split units need no zeroing: they carry
//             the call's epoch, see the chunk kernel),
// and stores the counts that the persistent kernels read.
// Pass 1 sums tokens, prefill tiles (W) and decode partial rows and finds the
// shortest and longest unit, which fix the run length, whether the partials fit
// the workspace (if not, nothing is split) and whether units are cut at all (see
// choose_split). Pass 2 walks the requests in chunks of 1024: one block scan
// gives each request its token and tile offsets, a second its list offsets, and
// a warp per request then writes that request's entries. Batches of at most 32
// requests and 8192 tokens (or of one request) take a one-warp kernel that
// builds the same lists without block barriers.
#include "common.cuh"
#include "plan.cuh"

namespace cpsa {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kScan = 6;

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

// KV tiles of one unit of query tile qt (rows [128 qt, 128 qt + rows)); see the
// tile grids in plan.cuh.
__device__ __forceinline__ int unit_tiles(const PlanParams &p, const Req &rq, int qt, int rows)
{
    return p.fused ? ceil_div(rq.hist, kTileN) + qt + 1 : ceil_div(rq.hist + qt * kTileM + rows, kTileN);
}

// Stream-K positions of all prefill units of one request: their KV tiles plus
// kUnitCostTiles per unit (0 for decode / invalid / empty).
__device__ int prefill_tiles(const PlanParams &p, const Req &rq)
{
    if (!rq.valid || rq.q < 2)
        return 0;
    const int units_per_qtile = p.Hkv * (p.group / p.nq);
    int tiles = 0;
    for (int qt = 0; qt * kTileM < rq.q; ++qt)
        tiles += (unit_tiles(p, rq, qt, min(kTileM, rq.q - qt * kTileM)) + kUnitCostTiles) * units_per_qtile;
    return tiles;
}

// Positions of the request's longest unit (its last query tile), 0 for decode /
// invalid / empty requests.
__device__ int longest_unit(const PlanParams &p, const Req &rq)
{
    if (!rq.valid || rq.q < 2)
        return 0;
    const int nqt = ceil_div(rq.q, kTileM);
    return unit_tiles(p, rq, nqt - 1, rq.q - (nqt - 1) * kTileM) + kUnitCostTiles;
}

// Positions of the request's shortest unit (its first query tile), INT_MAX for
// decode / invalid / empty requests.
__device__ int shortest_unit(const PlanParams &p, const Req &rq)
{
    if (!rq.valid || rq.q < 2)
        return 0x7fffffff;
    return unit_tiles(p, rq, 0, min(kTileM, rq.q)) + kUnitCostTiles;
}

__device__ int decode_splits(const Req &rq, int max_splits, int dec_heads)
{
    const int nch = ceil_div(rq.s, kDecodeChunk);
    int ns = ceil_div(rq.s, dec_heads > 1 ? kDecodeKeysPerSplitGrouped : kDecodeKeysPerSplit);
    ns = min(ns, max_splits);
    ns = min(ns, nch);
    return max(ns, 1);
}

// pieces; partial rows; combine units and combine items (split decode rows);
// decode items; split prefill units
struct Counts {
    int pieces, prows, cunits, citems, ditems, sunits;
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
// emit == true the entries are written at the given offsets, lane l of each pass
// taking one unit and placing its pieces by a warp scan.
// tile_off: global index of the request's first prefill tile; run: tiles per CTA
// run; cut: whether a run boundary may split a unit (else a unit goes whole to
// the run that holds its first tile).
__device__ Counts request_work(const PlanParams &p, int r, const Req &rq, int tile_off, int run, bool cut,
                               int max_splits, bool emit, int q_off, const Counts &off, int lane)
{
    Counts c{0, 0, 0, 0, 0, 0};
    if (!rq.valid || rq.q == 0)
        return c;
    if (rq.q == 1) {
        const int ns = decode_splits(rq, max_splits, p.dec_heads);
        const int nch = ceil_div(rq.s, kDecodeChunk);
        const int ngroups = p.Hkv / p.dec_heads;   // decode items per split
        c.ditems = ngroups * ns;
        if (ns > 1) {
            c.prows = p.Hq * ns;
            c.citems = 1;
            c.cunits = p.Hq;
        }
        if (emit) {
            for (int k = lane; k < c.ditems; k += 32) {
                const int sp = k / ngroups, kvh = k % ngroups;
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
    // prefill units in order: query tiles (longest KV range first), kv heads, head
    // pairs. Lane l of pass g0 takes unit g = g0 + l, the a-th query tile from the
    // last; its first tile is found in closed form (unit_tiles is hb + qt + 1 for
    // every query tile but the last, which may be short).
    static_assert(kTileM == kTileN, "unit tile counts assume square tiles");
    const int pairs = p.group / p.nq;
    const int upq = p.Hkv * pairs;            // units per query tile
    const int nqt = ceil_div(rq.q, kTileM);
    const int hb = ceil_div(rq.hist, kTileN);
    const int nkv_last = unit_tiles(p, rq, nqt - 1, rq.q - (nqt - 1) * kTileM);
    const int prow_unit = kTileM * p.nq;      // partial rows of one piece of a split unit
    const unsigned lanes_below = (1u << lane) - 1u;
    for (int g0 = 0; g0 < nqt * upq; g0 += 32) {
        const int g = g0 + lane;
        const bool active = g < nqt * upq;
        const int a = g / upq, j = g - a * upq;
        const int qt = nqt - 1 - a;
        const int nkv = a == 0 ? nkv_last : hb + qt + 1;
        // tiles of the units of query tiles nqt - 1 .. qt + 1: nkv_last, then hb + nqt - a' for a' = 1 .. a - 1
        const int before = a == 0 ? 0 : nkv_last + (a - 1) * (hb + nqt) - (a - 1) * a / 2;
        // the unit's positions [u0, u1): kUnitCostTiles of fixed cost, then its tiles from t0
        const int u0 = tile_off + upq * (before + a * kUnitCostTiles) + j * (nkv + kUnitCostTiles);
        const int t0 = u0 + kUnitCostTiles, u1 = t0 + nkv;
        const int first = t0 / run;
        const int np = active ? (cut ? (u1 - 1) / run - first + 1 : 1) : 0;
        const bool split = np > 1;
        // one scan for two sums: pieces (low word) and pieces of split units (high word)
        long long sc = (long long)np | ((long long)(split ? np : 0) << 32);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, sc, o);
            if (lane >= o) sc += y;
        }
        const long long tot = __shfl_sync(0xffffffffu, sc, 31);
        const long long ex = sc - ((long long)np | ((long long)(split ? np : 0) << 32));
        const unsigned split_lanes = __ballot_sync(0xffffffffu, split);
        if (emit && active) {
            const int kvh = j / pairs, hp = j - kvh * pairs;
            const int i0 = qt * kTileM;
            const int pi = off.pieces + c.pieces + (int)(ex & 0xffffffffll);
            // with cuts, every run starts a piece: the piece holding position c *
            // run (or the first one after it when that position is a unit's fixed
            // cost) is the first of CTA c's run
            if (!split) {
                p.pitems[pi] = PrefillItem{r, i0, kvh | (hp << 16), 0, nkv, (1 << 16), -1, first};
                if (cut && u0 <= first * run)
                    p.run_first[first] = pi;
            } else {
                // a split unit's partials: kTileM rows x nq heads x np pieces (see the chunk kernel's merge)
                const int pbase = off.prows + c.prows + prow_unit * (int)(ex >> 32);
                const int sunit = off.sunits + c.sunits + __popc(split_lanes & lanes_below);
                int x = t0;
                for (int pc = 0; pc < np; ++pc) {
                    const int owner = first + pc;
                    const int end = min(u1, (owner + 1) * run);
                    p.pitems[pi + pc] =
                        PrefillItem{r, i0, kvh | (hp << 16), x - t0, end - t0, pc | (np << 16), pbase, sunit};
                    if (pc > 0 || u0 <= owner * run)
                        p.run_first[owner] = pi + pc;
                    x = end;
                }
            }
        }
        c.pieces += (int)(tot & 0xffffffffll);
        c.sunits += __popc(split_lanes);
        c.prows += prow_unit * (int)(tot >> 32);
    }
    return c;
}

// Stream-K run length; cuts inside units only when splitting is allowed and the
// partials' bound fits the workspace (else nothing is split and the flag is set).
// A cut costs the run that holds it a second item and, at its end, a merge
// (about kCutCostTiles tiles of work, measured). When every unit is at least a
// run long, whole units land one per CTA (no run holds two unit starts) and cost
// the longest unit's length: then, if that is within kCutCostTiles of the run,
// nothing is cut.
struct SplitChoice {
    int run, max_splits;
    bool split_prefill, clamped;
};

__device__ SplitChoice choose_split(const PlanParams &p, long long tiles, int shortest, int longest,
                                    long long dprows)
{
    const int grid = max(1, p.chunk_grid);
    SplitChoice c;
    c.run = max((int)((tiles + grid - 1) / grid), kMinRunTiles);
    c.max_splits = p.max_splits;
    c.split_prefill = p.max_splits > 1;
    c.clamped = false;
    const long long pbound = (long long)2 * grid * kTileM * p.nq;
    if (p.max_splits > 1 && pbound + dprows > p.prow_capacity) {
        c.max_splits = 1;
        c.split_prefill = false;
        c.clamped = true;
    }
    if (c.split_prefill && shortest >= c.run && longest <= c.run + kCutCostTiles)
        c.split_prefill = false;
    return c;
}

// run_first[c] = first piece whose owner is >= c (pieces are sorted by owner);
// threads tid, tid + nthreads, ... of the caller share the entries. With cuts the
// emission already wrote the entries of runs holding tiles (runs [0, ceil(W /
// run))), and only the rest are set here; without cuts they are read back from
// the pieces' owners.
__device__ void fill_run_first(const PlanParams &p, int n_pieces, int grid, bool cut, long long tiles, int run,
                               int tid, int nthreads)
{
    if (cut) {
        const int first_empty = (int)((tiles + run - 1) / run);
        for (int c = first_empty + tid; c <= grid; c += nthreads) p.run_first[c] = n_pieces;
        return;
    }
    for (int i = tid; i <= n_pieces; i += nthreads) {
        const int lo = i == 0 ? 0 : p.pitems[i - 1].aux + 1;   // without cuts, aux is the owner CTA
        const int hi = i == n_pieces ? grid : p.pitems[i].aux;
        for (int c = lo; c <= hi; ++c) p.run_first[c] = i;
    }
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

// Block-wide maximum (hi) or minimum (!hi).
__device__ int block_extreme(int x, bool hi)
{
    __shared__ int red[kPlanThreads / 32];
    for (int o = 16; o > 0; o >>= 1) {
        const int y = __shfl_xor_sync(0xffffffffu, x, o);
        x = hi ? max(x, y) : min(x, y);
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
    __syncthreads();
    int m = red[0];
    for (int w = 1; w < kPlanThreads / 32; ++w) m = hi ? max(m, red[w]) : min(m, red[w]);
    __syncthreads();
    return m;
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
    // dependents are released at the end (see plan_small_kernel)
    pdl_wait();
    // ---- pass 1: tokens, prefill tiles, decode partial rows
    long long tok = 0, tiles = 0, dprows = 0;
    int longest = 0, shortest = 0x7fffffff;
    for (int base = 0; base < p.num_reqs; base += kPlanThreads) {
        const int r = base + threadIdx.x;
        if (r < p.num_reqs) {
            const Req rq = load_req(p, r);
            tok += rq.q > 0 ? rq.q : 0;   // invalid requests still occupy their rows
            tiles += prefill_tiles(p, rq);
            longest = max(longest, longest_unit(p, rq));
            shortest = min(shortest, shortest_unit(p, rq));
            if (rq.valid && rq.q == 1) {
                const int ns = decode_splits(rq, p.max_splits, p.dec_heads);
                if (ns > 1) dprows += (long long)p.Hq * ns;
            }
        }
    }
    tok = block_sum(tok);
    tiles = block_sum(tiles);
    dprows = block_sum(dprows);
    longest = block_extreme(longest, true);
    shortest = block_extreme(shortest, false);
    if (tok != p.num_tokens) {
        if (threadIdx.x == 0) set_dev_error(p.dev_err, CPSA_DEV_TOKENS_MISMATCH);
        if (threadIdx.x < kCntSlots) p.counts[threadIdx.x] = 0;
        for (int c = threadIdx.x; c <= p.chunk_grid; c += kPlanThreads) p.run_first[c] = 0;
        return;
    }
    const int grid = max(1, p.chunk_grid);
    const SplitChoice sc = choose_split(p, tiles, shortest, longest, dprows);
    const int run = sc.run, max_splits = sc.max_splits;
    const bool split_prefill = sc.split_prefill;
    if (sc.clamped && threadIdx.x == 0)
        set_dev_error(p.dev_err, CPSA_DEV_SPLITS_CLAMPED);

    // ---- pass 2: offsets and lists, 1024 requests at a time
    __shared__ int s_qoff[kPlanThreads], s_toff[kPlanThreads];
    __shared__ int s_cnt[kPlanThreads][kScan];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int carry_a[2] = {0, 0};                        // tokens, tiles
    int carry_b[kScan] = {0, 0, 0, 0, 0, 0};        // pieces, prows, cunits, citems, ditems, sunits
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
                                          s_qoff[l], Counts{0, 0, 0, 0, 0, 0}, lane);
            if (lane == 0) {
                s_cnt[l][0] = c.pieces;
                s_cnt[l][1] = c.prows;
                s_cnt[l][2] = c.cunits;
                s_cnt[l][3] = c.citems;
                s_cnt[l][4] = c.ditems;
                s_cnt[l][5] = c.sunits;
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
            const Counts off{s_cnt[l][0], s_cnt[l][1], s_cnt[l][2], s_cnt[l][3], s_cnt[l][4], s_cnt[l][5]};
            request_work(p, base + l, rq, s_toff[l], run, split_prefill, max_splits, true, s_qoff[l], off, lane);
        }
        __syncthreads();
    }
    __syncthreads();   // this block's piece writes are visible to the whole block
    const int n_pieces = (int)min((int64_t)carry_b[0], p.max_pitems);
    fill_run_first(p, n_pieces, grid, split_prefill, tiles, run, threadIdx.x, kPlanThreads);
    if (threadIdx.x == 0) {
        p.cu_q[p.num_reqs] = carry_a[0];
        p.counts[kCntPrefill] = (int)min((int64_t)carry_b[0], p.max_pitems);
        p.counts[kCntCombine] = (int)min((int64_t)carry_b[3], p.max_citems);
        p.counts[kCntPartialRows] = carry_b[1];
        p.counts[kCntCombineUnits] = carry_b[2];
        p.counts[kCntDecode] = (int)min((int64_t)carry_b[4], p.max_ditems);
        p.counts[kCntRunTiles] = run;
        p.counts[kCntSplitUnits] = carry_b[5];
        for (int j = kCntSplitUnits + 1; j < kCntSlots; ++j) p.counts[j] = 0;
    }
    pdl_trigger();
}

// The same lists for a batch of at most 32 requests, built by one warp: lane r
// holds request r, warp scans give the token and tile offsets, and the warp then
// walks the requests in order, so every request's list offsets are the running
// totals of the ones before it (one pass, no block-wide barriers).
__global__ void __launch_bounds__(32, 1) plan_small_kernel(PlanParams p)
{
    // The attention kernels that follow are released only at the end: CTAs
    // launched early wait beside this warp and halve its speed (measured), while
    // what they would overlap is short.
    pdl_wait();
    const int lane = threadIdx.x;
    const bool mine = lane < p.num_reqs;
    Req rq{false, 0, 0, 0};
    if (mine)
        rq = load_req(p, lane);
    const int tok = mine && rq.q > 0 ? rq.q : 0;   // invalid requests still occupy their rows
    const int tiles = mine ? prefill_tiles(p, rq) : 0;
    int longest = mine ? longest_unit(p, rq) : 0;
    int shortest = mine ? shortest_unit(p, rq) : 0x7fffffff;
    int dprows = 0;
    if (mine && rq.valid && rq.q == 1) {
        const int ns = decode_splits(rq, p.max_splits, p.dec_heads);
        if (ns > 1) dprows = p.Hq * ns;
    }
    // totals in 64 bits first: the 32-bit scans below are only used once they fit
    long long tok_sum = tok, tile_sum = tiles, dprow_sum = dprows;
    for (int o = 16; o > 0; o >>= 1) {
        longest = max(longest, __shfl_xor_sync(0xffffffffu, longest, o));
        shortest = min(shortest, __shfl_xor_sync(0xffffffffu, shortest, o));
        tok_sum += __shfl_xor_sync(0xffffffffu, tok_sum, o);
        tile_sum += __shfl_xor_sync(0xffffffffu, tile_sum, o);
        dprow_sum += __shfl_xor_sync(0xffffffffu, dprow_sum, o);
    }
    const int grid = max(1, p.chunk_grid);
    if (tok_sum != p.num_tokens) {
        if (lane == 0) set_dev_error(p.dev_err, CPSA_DEV_TOKENS_MISMATCH);
        if (lane < kCntSlots) p.counts[lane] = 0;
        for (int c = lane; c <= p.chunk_grid; c += 32) p.run_first[c] = 0;
        return;
    }
    if (mine && !rq.valid)
        set_dev_error(p.dev_err, (rq.q < 0 || rq.s < rq.q) ? CPSA_DEV_SEQ_LT_QUERY : CPSA_DEV_SEQ_GT_TABLE);
    int tok_total, tile_total;
    const int tok_off = warp_excl_scan(tok, lane, tok_total);
    const int tile_off = warp_excl_scan(tiles, lane, tile_total);
    if (mine)
        p.cu_q[lane] = tok_off;
    const SplitChoice sc = choose_split(p, tile_sum, shortest, longest, dprow_sum);
    if (sc.clamped && lane == 0)
        set_dev_error(p.dev_err, CPSA_DEV_SPLITS_CLAMPED);
    Counts off{0, 0, 0, 0, 0, 0};
    for (int r = 0; r < p.num_reqs; ++r) {
        Req rr;
        rr.valid = __shfl_sync(0xffffffffu, rq.valid ? 1 : 0, r) != 0;
        rr.q = __shfl_sync(0xffffffffu, rq.q, r);
        rr.s = __shfl_sync(0xffffffffu, rq.s, r);
        rr.hist = __shfl_sync(0xffffffffu, rq.hist, r);
        const int qoff = __shfl_sync(0xffffffffu, tok_off, r);
        const int toff = __shfl_sync(0xffffffffu, tile_off, r);
        const Counts c = request_work(p, r, rr, toff, sc.run, sc.split_prefill, sc.max_splits, true, qoff, off, lane);
        off.pieces += c.pieces;
        off.prows += c.prows;
        off.cunits += c.cunits;
        off.citems += c.citems;
        off.ditems += c.ditems;
        off.sunits += c.sunits;
    }
    __syncwarp();   // the warp's piece writes are visible to all its lanes
    const int n_pieces = (int)min((int64_t)off.pieces, p.max_pitems);
    fill_run_first(p, n_pieces, grid, sc.split_prefill, tile_sum, sc.run, lane, 32);
    if (lane == 0) {
        p.cu_q[p.num_reqs] = tok_total;
        p.counts[kCntPrefill] = n_pieces;
        p.counts[kCntCombine] = (int)min((int64_t)off.citems, p.max_citems);
        p.counts[kCntPartialRows] = off.prows;
        p.counts[kCntCombineUnits] = off.cunits;
        p.counts[kCntDecode] = (int)min((int64_t)off.ditems, p.max_ditems);
        p.counts[kCntRunTiles] = sc.run;
        p.counts[kCntSplitUnits] = off.sunits;
    } else if (lane > kCntSplitUnits && lane < kCntSlots) {
        p.counts[lane] = 0;
    }
    pdl_trigger();
}

}  // namespace

// The one-warp kernel walks every request's units itself (about 0.5 us per 32
// units: 166 us for 32 prompts of 2600 tokens at 32/8 heads), the block kernel
// gives each request a warp of its own but pays its barriers: one warp while
// the lists are short or there is one request to walk.
constexpr int64_t kPlanSmallMaxTokens = 8192;

cudaError_t launch_plan(const PlanParams &p, cudaStream_t s, bool early)
{
    if (p.num_reqs <= 32 && (p.num_reqs == 1 || p.num_tokens <= kPlanSmallMaxTokens))
        return launch_pdl(early, plan_small_kernel, dim3(1), dim3(32), 0, s, p);
    return launch_pdl(early, plan_kernel, dim3(1), dim3(kPlanThreads), 0, s, p);
}

}  // namespace cpsa
