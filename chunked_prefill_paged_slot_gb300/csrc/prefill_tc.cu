// prefill_tc.cu -- causal chunked-prefill attention on the 5th-generation tensor
// cores (tcgen05 + TMEM), K/V tiles gathered page by page from the paged cache
// with TMA.
//
// What it computes ("vLLM Chunked-Prefills" article, section 3.2.1, chunked
// attention; metadata from the "Ascend dual-stream parallel" article, section
// 3.1): for a 128-row tile of one request's new tokens and NQ q heads that share
// one kv head, softmax(scale * Q K^T) V over the keys 0 .. h_r + i of every row i,
// the history keys read from the cache pages listed in block_table. The chunk's
// own keys come from the cache too, or, with the KV write fused (the KV write
// of the dual-stream article's section 3.1 folded into this kernel), straight
// from the new K/V rows, each tile of them also stored once to its cache slots.
//
// CTA layout (352 threads, one CTA per SM, persistent over prefill items):
//   warp 8       TMA producer: Q tiles once per item, then K_j, V_j into a ring
//                of shared-memory slots (one box per page and 64-column half;
//                below page 128 a cache V tile takes one box per page holding
//                both halves, page-major in the slot); block_table lookups;
//                zeroes the value rows past the tile's last key (they may hold
//                anything).
//   warp 9       tcgen05 issuer (one elected lane per instruction, the warp
//                converged): S_n = Q_n K_j^T into TMEM, then O_n += P_n V_j with
//                P_n read from TMEM; TMEM alloc/dealloc.
//   warps 0..7   softmax, one warpgroup per q head n; thread = query row:
//                S row from TMEM (the reducing load gives the row max of an
//                unmasked tile), causal mask on the diagonal/tail tiles, online
//                max/sum in fp32 (base-2 exponent, scale folded in), P as bf16
//                back into TMEM over S; final O / l epilogue (planned batches
//                without the KV write: staged in shared memory, TMA stores), or for a piece of
//                a unit cut by the stream-K split, its partial (O / l in bf16,
//                m and l in fp32) or the merge of all the unit's pieces
//                (whichever piece finishes last merges; at the end of a run
//                through the then idle Q and K/V buffers).
//   warp 10      cache writer (fused KV write only): for each tile of new rows
//                this CTA owns (the diagonal tile of head pair 0), TMA-loads its
//                K and then its V rows into a staging buffer of its own and
//                TMA-stores them to the cache pages slot_mapping names, apart
//                from the attention pipeline (rows whose slots do not form whole
//                page boxes are stored row by row).
// Exponentials: MUFU ex2. A build-time knob (kFmaExpPairsPer8, 0 by default:
// measured fastest on GB300) sends that many of every 8 pairs of an unmasked
// tile to the FMA pipe instead (exp2_poly_x2). The row sum and the exponent
// arguments use packed f32x2 arithmetic.
// Rescaling of O is lazy: the running maximum is only raised when a tile's
// maximum exceeds it by more than 8 (a factor 256 in the exponent), which keeps
// p <= 256 and leaves the final O / l unchanged.
// TMEM columns: S_0 [0,128) S_1 [128,256) O_0 [256,256+D) O_1 [256+D, 256+2D).
#include "common.cuh"
#include "kernels.cuh"
#include "plan.cuh"

namespace cpsa {

namespace {

// Of every 8 exponent pairs of an unmasked S row, this many go to the FMA pipe.
#ifndef CPSA_FMA_EXP_PAIRS_PER_8
#define CPSA_FMA_EXP_PAIRS_PER_8 0   // measured fastest on GB300: MUFU keeps up on this kernel
#endif
constexpr int kFmaExpPairsPer8 = CPSA_FMA_EXP_PAIRS_PER_8;

// The merge of split units (merge_split_row): pieces besides the merging one,
// and the shared memory each softmax warp takes for their bf16 partials when it
// stages them (others x 32 rows x 128 columns x 2 B).
constexpr int kMergeMaxOthers = 3;
constexpr int kMergeStageBytes = kMergeMaxOthers * 32 * 128 * 2;

template <int D, int NQ>
struct ChunkCfg {
    static constexpr int kHalves = D / 64;             // 128-byte swizzle atoms across a row
    static constexpr int kHalfBytes = 128 * 128;       // 128 rows x 64 bf16
    static constexpr int kTileBytes = kHalves * kHalfBytes;
    static constexpr int kSlots = D == 128 ? 4 : 8;
    static constexpr int kQOff = 0;
    static constexpr int kSlotOff = NQ * kTileBytes;
    static constexpr int kStageOff = kSlotOff + kSlots * kTileBytes;   // the cache writer's buffer
    static constexpr int kBarOff = kStageOff + kTileBytes;
    static constexpr int kItemOff = kBarOff + 256;             // self-planned pieces (after ChunkBars)
    static constexpr int kBarBytes = 256 + kSelfPlanCap * 32;  // barriers + pieces
    static constexpr int kSmemBytes = kBarOff + kBarBytes + 1024;   // + alignment slack
    static_assert(kSmemBytes <= 232448, "beyond the 227 KB of shared memory a CTA may have");
    static_assert(D != 128 || NQ * 4 * kMergeStageBytes <= kSlotOff + kSlots * kTileBytes,
                  "the staged merge uses the Q and K/V buffers");
    static constexpr int kThreads = 352;
    static constexpr int kLoadWarp = 8;
    static constexpr int kMmaWarp = 9;
    static constexpr int kWriteWarp = 10;
    static constexpr uint32_t kTmemCols = 512;
    __host__ __device__ static constexpr uint32_t s_col(int n) { return (uint32_t)n * 128u; }
    __host__ __device__ static constexpr uint32_t o_col(int n) { return 256u + (uint32_t)n * D; }
};

struct ChunkBars {
    uint64_t q_full, q_empty, tail, drain;
    uint64_t s_full[2], p_full[2], o_done[2];
    uint64_t slot_full[8], slot_empty[8];
    uint64_t stage;        // fused KV write: the writer's buffer is loaded
    uint64_t writer_done;  // the cache writer has finished with its buffer (its last store has read it)
    uint32_t tmem_base;
    int abort;
    int it_begin, it_end;    // this CTA's run of pieces
};
static_assert(sizeof(ChunkBars) <= 256, "the self-planned pieces follow the barriers at +256");
static_assert(sizeof(PrefillItem) == 32, "piece size");

// Merge counters carry the call's epoch in their high 32 bits (see ChunkParams)
// and are cleared by the warp that merges, so a counter holds another call's
// count only after a call that ended early (a device error).
__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed_gpu_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Pieces of this call counted in a counter (0 when it still holds an earlier call's count).
__device__ __forceinline__ int epoch_count(unsigned long long v, uint32_t epoch)
{
    return (uint32_t)(v >> 32) == epoch ? (int)(uint32_t)v : 0;
}

// Counts one more piece of this call and returns the count before it (a counter
// left by an earlier call starts over at one). `old` is the caller's earlier
// read of the counter, the first guess of the exchange (read before the
// partial's stores, its latency overlaps them). An exchange fails only when the
// guess was stale or another piece counted itself in between, so the loop ends
// within a few more rounds than the unit has pieces; the cap is a safeguard that
// flags an error rather than spin.
__device__ __forceinline__ int epoch_arrive(unsigned long long *cnt, uint32_t epoch, unsigned long long old,
                                            uint32_t *dev_err)
{
    for (int i = 0; i < 4096; ++i) {
        const bool cur = (uint32_t)(old >> 32) == epoch;
        const unsigned long long nv = cur ? old + 1ull : (((unsigned long long)epoch << 32) | 1ull);
        const unsigned long long prev = atomicCAS(cnt, old, nv);
        if (prev == old)
            return cur ? (int)(uint32_t)old : 0;
        old = prev;
    }
    set_dev_error(dev_err, CPSA_DEV_WAIT_TIMEOUT);
    return -1;
}

// The units of a self-planned batch that fall in this CTA's run (see
// self_plan_run); I is the integer type of the tile positions: 32 bits whenever
// the request's W tiles fit (64-bit division is a long software routine on the
// GPU, and this walk sits on every launch's critical path), 64 bits otherwise.
template <int NQ, typename I>
__device__ __forceinline__ int self_plan_walk(PrefillItem *items, int lane, int nqt, int hb, int nkv_last, int upq,
                                              int pairs, I run, bool cut)
{
    const I lo = (I)blockIdx.x * run, hi = lo + run;
    const int prow_unit = kTileM * NQ;
    const unsigned below = (1u << lane) - 1u;
    const int G = nqt * upq;
    int n = 0;
    for (int g0 = 0; g0 < G; g0 += 32) {
        const int g = g0 + lane;
        const bool active = g < G;
        const int a = g / upq, j = g - a * upq;
        const int qt = nqt - 1 - a;
        const int nkv = a == 0 ? nkv_last : hb + qt + 1;
        // KV tiles of one unit column before the a-th query tile from the last
        const I before = a == 0 ? (I)0 : (I)nkv_last + (I)(a - 1) * (I)(hb + nqt) - (I)((a - 1) * a / 2);
        // the unit's positions: kUnitCostTiles of fixed cost from u0, its tiles [t0, u1)
        const I u0 = (I)upq * (before + (I)a * kUnitCostTiles) + (I)j * (I)(nkv + kUnitCostTiles);
        const I t0 = u0 + kUnitCostTiles, u1 = t0 + (I)nkv;
        // with cuts a run takes every piece of a unit inside it; without, whole units
        // go to the run that holds their first tile
        const bool take = active && (cut ? (u1 > lo && t0 < hi) : (t0 >= lo && t0 < hi));
        const unsigned m = __ballot_sync(0xffffffffu, take);
        if (take) {
            const int k = n + __popc(m & below);
            if (k < kSelfPlanCap) {
                const int kvh = j / pairs, hp = j - kvh * pairs;
                const I c0 = t0 / run;
                const int np = cut ? (int)((u1 - 1) / run - c0 + 1) : 1;
                if (np == 1) {
                    items[k] = PrefillItem{0, qt * kTileM, kvh | (hp << 16), 0, nkv, 1 << 16, -1, (int)blockIdx.x};
                } else {
                    const I x0 = t0 > lo ? t0 : lo, x1 = u1 < hi ? u1 : hi;
                    items[k] = PrefillItem{0, qt * kTileM, kvh | (hp << 16), (int)(x0 - t0), (int)(x1 - t0),
                                           ((int)blockIdx.x - (int)c0) | (np << 16), 2 * (int)c0 * prow_unit,
                                           (int)c0};
                }
            }
        }
        n += __popc(m);
        // units come in tile order: after one whose tiles start at or past the run's
        // end, none is in it
        if (__shfl_sync(0xffffffffu, active ? (t0 >= hi ? 1 : 0) : 1, 31))
            break;
    }
    return n;
}

// The pieces of this CTA's stream-K run for a batch of one prefill request,
// computed by the CTA itself (one warp) instead of the plan kernel. Units,
// their order (query tiles from the last, then kv heads, then head pairs), the
// run length, the rule for cutting units and the piece fields are the plan's
// (plan.cu: request_work, choose_split). Only the addresses of a split unit's
// partial rows and merge counters differ: they follow from the run c0 that holds
// the unit's first tile, rows [2 c0, 2 c0 + np) x (128 NQ) and counter c0,
// instead of from its rank among split units (which needs the whole list). A
// run holds at most one piece that continues a split unit (its first) and at
// most one that starts one (its last), so a later split unit starts in run
// c0' >= c0 + np - 1 and its rows begin at 2 c0' >= 2 c0 + 2 np - 2 >= 2 c0 + np
// (np >= 2): no overlap, and 2 x grid x 128 NQ rows are enough (the host checks
// that they fit before it allows cuts). A piece of run c belongs to it, so its
// index within its unit is c - c0. Validation as in the plan, flags raised by
// CTA 0. Writes up to kSelfPlanCap pieces; returns their number (warp-uniform).
// Everything the self plan reads from the kernel's parameters, passed by value:
// the plan lives out of line (so that its registers do not weigh on the softmax
// and MMA loops, which sit at the register cap), and a reference to the
// parameter block would make every thread copy the block to local memory.
struct SelfPlanArgs {
    const int32_t *query_lens, *seq_lens;
    uint32_t *dev_err;
    int num_tokens, max_blocks, page_size, group, num_kv_heads, fused, split_ok, split_clamped;
};

template <int NQ>
__device__ __noinline__ int self_plan_run(const SelfPlanArgs a, PrefillItem *items, int lane)
{
    const int q = __ldg(a.query_lens), s = __ldg(a.seq_lens);
    uint32_t bad = 0;
    if (q != a.num_tokens)
        bad = CPSA_DEV_TOKENS_MISMATCH;
    else if (q < 0 || s < q)
        bad = CPSA_DEV_SEQ_LT_QUERY;
    else if ((int64_t)s > (int64_t)a.max_blocks * a.page_size)
        bad = CPSA_DEV_SEQ_GT_TABLE;
    if (blockIdx.x == 0 && lane == 0) {
        if (bad)
            set_dev_error(a.dev_err, bad);
        if (a.split_clamped)
            set_dev_error(a.dev_err, CPSA_DEV_SPLITS_CLAMPED);
    }
    if (bad || q < 2)
        return 0;
    const int hist = s - q;
    const int pairs = a.group / NQ;
    const int upq = a.num_kv_heads * pairs;      // units per query tile
    const int nqt = (q + kTileM - 1) / kTileM;
    const int hb = (hist + kTileN - 1) / kTileN;
    const int nkv_last = a.fused ? hb + nqt : (hist + q + kTileN - 1) / kTileN;
    const long long W = (long long)upq * (nkv_last + (long long)(nqt - 1) * (hb + nqt) - (long long)(nqt - 1) * nqt / 2 +
                                          (long long)nqt * kUnitCostTiles);
    const int shortest = (nqt == 1 ? nkv_last : hb + 1) + kUnitCostTiles;
    const long long grid = gridDim.x;
    const long long run = max((W + grid - 1) / grid, (long long)kMinRunTiles);
    const bool cut = a.split_ok && !(shortest >= run && nkv_last + kUnitCostTiles <= run + kCutCostTiles);
    int n = W + run < 0x7fffffffll
                ? self_plan_walk<NQ, int>(items, lane, nqt, hb, nkv_last, upq, pairs, (int)run, cut)
                : self_plan_walk<NQ, long long>(items, lane, nqt, hb, nkv_last, upq, pairs, run, cut);
    if (n > kSelfPlanCap) {
        if (lane == 0)
            set_dev_error(a.dev_err, CPSA_DEV_PLAN_OVERFLOW);
        n = kSelfPlanCap;
    }
    return n;
}

// Cache stores of one staged K or V tile of new rows (128 rows, 128-byte
// swizzled 64-column halves), rows [0, rows) to the slots sl of kv head kvh (lane
// l holds the slots of rows l, l + 32, l + 64, l + 96). The tile is cut into
// boxes of PB = min(page_size, 128) rows; a box whose rows are valid tokens with
// consecutive slots inside one page is stored by TMA through the cache's own
// tensor map (box_mask bit j, box start slots in s0), the rest row by row from
// shared memory (lane = row, no shuffles). Negative slots are padding; slots past
// the cache set the error flag. Lane 0 commits the TMA stores as one bulk group.
template <int D>
__device__ __forceinline__ void store_tile_rows(const ChunkParams &p, const CUtensorMap *map, const uint8_t *tile,
                                                void *cache, int kvh, int rows, const int64_t (&sl)[4],
                                                uint32_t box_mask, const int64_t *s0, int PB, int lane,
                                                bool flag_errors)
{
    constexpr int CPR = D / 8;        // 16-byte chunks per row
    const int lg_p = __ffs(p.page_size) - 1;   // page_size is a power of two
    const int64_t n_slots = p.num_pages * (int64_t)p.page_size;
    if (lane == 0) {
        for (int j = 0; j < 128 / PB; ++j) {
            if (!((box_mask >> j) & 1u))
                continue;
            const int off = (int)(s0[j] & (p.page_size - 1));
            const int z = (int)((s0[j] >> lg_p) * p.num_kv_heads + kvh);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
                tma_store_3d(map, tile + c * (128 * 128) + j * PB * 128, c * 64, off, z);
        }
        bulk_commit_group();
    }
    uint4 *dst_base = reinterpret_cast<uint4 *>(cache);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int row = lane + 32 * q;
        const int64_t slot = sl[q];
        if (row >= rows || slot < 0 || ((box_mask >> (row / PB)) & 1u))
            continue;
        if (slot >= n_slots) {
            if (flag_errors)
                set_dev_error(p.dev_err, CPSA_DEV_SLOT_OUT_OF_RANGE);
            continue;
        }
        uint4 *dst = dst_base + (((slot >> lg_p) * p.num_kv_heads + kvh) * p.page_size +
                                 (slot & (p.page_size - 1))) * CPR;
#pragma unroll 4
        for (int ch = 0; ch < CPR; ++ch)
            dst[ch] = *reinterpret_cast<const uint4 *>(tile + (ch >> 3) * (128 * 128) + row * 128 +
                                                       (((ch & 7) ^ (row & 7)) << 4));
    }
}

// The merge of a split unit's row (see the epilogue): sums in piece order, this
// piece's own terms (its TMEM O, m, l) taken at its place, so the bits do not
// depend on which piece merges; writes the bf16 row. Kept out of line so that
// its registers do not weigh on the softmax loop.
// bf16 of x, back in fp32 (round to nearest even, as pack_bf16x2)
__device__ __forceinline__ float bf16_round(float x)
{
    return __uint_as_float(pack_bf16x2(x, 0.f) << 16);
}

__device__ __forceinline__ void bf16x8_unpack(const uint4 &u, float *v)
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        v[2 * k] = __uint_as_float(w[k] << 16);
        v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
}

// (m, l) of every piece of a split unit's row and the weights of the merge:
// out = sum_q wq[q] * Ohat_q / L with wq[q] = 2^(m_q - M) l_q, L = sum_q wq[q],
// Ohat_q = O_q / l_q as stored (bf16). At most kMergeMaxOthers + 1 pieces.
template <int NQ>
__device__ __forceinline__ float merge_weights(const float2 *pml, int piece, int npieces, int wg, int row, float m_use,
                                               float l, float (&wq)[kMergeMaxOthers + 1])
{
    float mq[kMergeMaxOthers + 1], lq[kMergeMaxOthers + 1];
    float M = m_use;
#pragma unroll
    for (int q = 0; q <= kMergeMaxOthers; ++q) {
        mq[q] = m_use;
        lq[q] = l;
        if (q < npieces && q != piece) {
            const float2 ml = __ldcg(pml + (q * NQ + wg) * 128 + row);
            mq[q] = ml.x;
            lq[q] = ml.y;
            M = fmaxf(M, ml.x);
        }
    }
    const float Mref = M == -INFINITY ? 0.f : M;
    float L = 0.f;
#pragma unroll
    for (int q = 0; q <= kMergeMaxOthers; ++q) {
        wq[q] = ex2_approx(mq[q] - Mref) * lq[q];
        if (q < npieces)
            L += wq[q];
    }
    return L > 0.f ? 1.f / L : 0.f;
}

// The merge of a split unit's row (see the epilogue): every piece's normalized
// partial Ohat_q (this piece's own from its TMEM O, rounded to bf16 exactly as it
// would have been stored) weighted in piece order, so the bits do not depend on
// which piece merges; writes the bf16 row. Up to kMergeMaxOthers + 1 pieces.
// The other pieces' partials come either straight from L2 (stage == nullptr) or,
// at the end of a CTA's run when the Q and K/V buffers are free, all at once
// through this warp's kMergeStageBytes of them (cp.async), so the L2 latency is
// paid once. Kept out of line so that its registers do not weigh on the softmax
// loop.
//
// The weighted sum runs on packed f32x2 pairs (one fma.rn.f32x2 per pair and
// piece, the rounding of one fmaf per element, in the same order). With ostage
// (this warp's 4 KB of the cache writer's buffer, free at the end of a run) and
// every row valid, the merged rows leave by TMA stores through the `out` map,
// 64 columns at a time; otherwise each lane stores its row.
template <int D, int NQ>
__device__ __noinline__ void merge_split_row(const ChunkParams &p, uint32_t tO, const float2 *pml, const uint4 *ph,
                                             int piece, int npieces, int wg, int row, int lane, float m_use, float l,
                                             bool valid_row, int64_t out_off, uint4 *stage, uint8_t *ostage,
                                             const CUtensorMap *tm_o, int h, int t_row0)
{
    float wq[kMergeMaxOthers + 1];
    const float inv_L = merge_weights<NQ>(pml, piece, npieces, wg, row, m_use, l, wq);
    const float inv_own = l > 0.f ? 1.f / l : 0.f;
    const bool staged_out = ostage != nullptr && __all_sync(0xffffffffu, valid_row);
    if (stage != nullptr) {
#pragma unroll
        for (int q = 0; q <= kMergeMaxOthers; ++q) {
            if (q < npieces && q != piece) {
                const int qi = q - (q > piece ? 1 : 0);
                const uint4 *src = ph + (int64_t)(q * NQ + wg) * (D / 8) * 128 + row;
#pragma unroll
                for (int j = 0; j < D / 8; ++j) cp_async_cg16(stage + (qi * (D / 8) + j) * 32 + lane, src + j * 128);
            }
        }
        cp_async_wait_all();
    }
    // bf16 pair (low half first) as an f32x2 pair
    auto widen = [](uint32_t w) -> uint64_t { return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)); };
    const uint64_t own2 = f2_pack(inv_own, inv_own), invL2 = f2_pack(inv_L, inv_L);
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tO + c * 32, r);
        tmem_wait_ld();
        uint64_t acc[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) acc[x] = 0ull;
#pragma unroll
        for (int q = 0; q <= kMergeMaxOthers; ++q) {
            if (q >= npieces)
                continue;
            const uint64_t w2 = f2_pack(wq[q], wq[q]);
            if (q == piece) {
                // this piece's O / l rounded to bf16 like the stored partials
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    float a, b;
                    f2_unpack(f2_mul(f2_pack(__uint_as_float(r[2 * x]), __uint_as_float(r[2 * x + 1])), own2), a, b);
                    acc[x] = f2_fma(widen(pack_bf16x2(a, b)), w2, acc[x]);
                }
            } else {
                const int qi = q - (q > piece ? 1 : 0);
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const uint4 u = stage != nullptr
                                        ? stage[(qi * (D / 8) + c * 4 + x) * 32 + lane]
                                        : __ldcg(ph + ((int64_t)(q * NQ + wg) * (D / 8) + c * 4 + x) * 128 + row);
                    acc[4 * x + 0] = f2_fma(widen(u.x), w2, acc[4 * x + 0]);
                    acc[4 * x + 1] = f2_fma(widen(u.y), w2, acc[4 * x + 1]);
                    acc[4 * x + 2] = f2_fma(widen(u.z), w2, acc[4 * x + 2]);
                    acc[4 * x + 3] = f2_fma(widen(u.w), w2, acc[4 * x + 3]);
                }
            }
        }
        uint32_t pk[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) {
            float a, b;
            f2_unpack(f2_mul(acc[x], invL2), a, b);
            pk[x] = pack_bf16x2(a, b);
        }
        if (staged_out) {
            // 64 columns per store: blocks c = 2 c2 and 2 c2 + 1, row `lane` at lane * 128
            // bytes, 16-byte chunk j at (j ^ (lane & 7)) (the map's 128-byte swizzle)
            if ((c & 1) == 0) {
                if (lane == 0)
                    bulk_wait_group_read0();   // the previous store has read the buffer
                __syncwarp();
            }
#pragma unroll
            for (int x = 0; x < 4; ++x)
                *reinterpret_cast<uint4 *>(ostage + lane * 128 + ((((c & 1) * 4 + x) ^ (lane & 7)) << 4)) =
                    make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
            if ((c & 1) == 1) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(tm_o, ostage, (c >> 1) * 64, h, t_row0);
                    bulk_commit_group();
                }
            }
        } else if (valid_row) {
            uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + out_off + c * 32);
#pragma unroll
            for (int x = 0; x < 4; ++x)
                dst[x] = make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
        }
    }
}

// The rows of a whole unit in the self-planned kernel without the KV write: as
// in the planned kernel's epilogue, each warp stages its 32 rows, 64 columns at
// a time, in its own 4 KB (stg) of the cache writer's idle buffer and a TMA
// store writes them out; a warp with rows past the request's end stores its
// valid rows directly. Out of line: compiled into the self-planned kernel's
// loop, the same code measured slower on one-request chunks with the KV write
// fused, which never take it.
template <int D>
__device__ __noinline__ void store_unit_rows_staged(uint32_t tO, float l, bool valid_row, uint8_t *stg,
                                                    const CUtensorMap *tm_o, __nv_bfloat16 *out, int64_t t_row,
                                                    int h, int num_q_heads, int lane)
{
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    const bool staged = __all_sync(0xffffffffu, valid_row);
#pragma unroll
    for (int c2 = 0; c2 < D / 64; ++c2) {
        // 64 columns into registers first: the wait for the previous store's read
        // (the other half's, just issued) overlaps the TMEM loads
        uint4 v[2][4];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            uint32_t r[32];
            tmem_ld32(tO + (2 * c2 + cc) * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int x = 0; x < 4; ++x)
                v[cc][x] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * x + 0]) * inv_l, __uint_as_float(r[8 * x + 1]) * inv_l),
                                      pack_bf16x2(__uint_as_float(r[8 * x + 2]) * inv_l, __uint_as_float(r[8 * x + 3]) * inv_l),
                                      pack_bf16x2(__uint_as_float(r[8 * x + 4]) * inv_l, __uint_as_float(r[8 * x + 5]) * inv_l),
                                      pack_bf16x2(__uint_as_float(r[8 * x + 6]) * inv_l, __uint_as_float(r[8 * x + 7]) * inv_l));
        }
        if (staged) {
            if (lane == 0)
                bulk_wait_group_read0();   // the warp's previous store has read the buffer
            __syncwarp();
#pragma unroll
            for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                for (int x = 0; x < 4; ++x)
                    *reinterpret_cast<uint4 *>(stg + lane * 128 + (((cc * 4 + x) ^ (lane & 7)) << 4)) = v[cc][x];
        } else if (valid_row) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint4 *dst = reinterpret_cast<uint4 *>(out + (t_row * num_q_heads + h) * D + (2 * c2 + cc) * 32);
#pragma unroll
                for (int x = 0; x < 4; ++x)
                    dst[x] = v[cc][x];
            }
        }
        if (staged) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_3d(tm_o, stg, c2 * 64, h, (int)(t_row - lane));
                bulk_commit_group();
            }
        }
    }
}

// The same merge for units of more than kMergeMaxOthers + 1 pieces (long KV
// ranges against short runs), every partial straight from L2; the same weights,
// order and rounding as merge_split_row.
template <int D, int NQ>
__device__ __noinline__ void merge_split_row_any(const ChunkParams &p, uint32_t tO, const float2 *pml, const uint4 *ph,
                                                 int piece, int npieces, int wg, int row, float m_use, float l,
                                                 bool valid_row, int64_t out_off)
{
    float M = m_use;
    for (int q = 0; q < npieces; ++q)
        if (q != piece)
            M = fmaxf(M, __ldcg(pml + (q * NQ + wg) * 128 + row).x);
    const float Mref = M == -INFINITY ? 0.f : M;
    float L = 0.f;
    for (int q = 0; q < npieces; ++q) {
        const float2 ml = q == piece ? make_float2(m_use, l) : __ldcg(pml + (q * NQ + wg) * 128 + row);
        L += ex2_approx(ml.x - Mref) * ml.y;
    }
    const float inv_L = L > 0.f ? 1.f / L : 0.f;
    const float inv_own = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tO + c * 32, r);
        tmem_wait_ld();
        float acc[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) acc[x] = 0.f;
        for (int q = 0; q < npieces; ++q) {
            float v[32];
            float2 ml;
            if (q == piece) {
                ml = make_float2(m_use, l);
#pragma unroll
                for (int x = 0; x < 32; ++x) v[x] = bf16_round(__uint_as_float(r[x]) * inv_own);
            } else {
                ml = __ldcg(pml + (q * NQ + wg) * 128 + row);
#pragma unroll
                for (int x = 0; x < 4; ++x)
                    bf16x8_unpack(__ldcg(ph + ((int64_t)(q * NQ + wg) * (D / 8) + c * 4 + x) * 128 + row), v + 8 * x);
            }
            const float wq = ex2_approx(ml.x - Mref) * ml.y;
#pragma unroll
            for (int x = 0; x < 32; ++x) acc[x] = fmaf(wq, v[x], acc[x]);
        }
        if (valid_row) {
            uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + out_off + c * 32);
#pragma unroll
            for (int x = 0; x < 4; ++x)
                dst[x] = make_uint4(pack_bf16x2(acc[8 * x + 0] * inv_L, acc[8 * x + 1] * inv_L),
                                    pack_bf16x2(acc[8 * x + 2] * inv_L, acc[8 * x + 3] * inv_L),
                                    pack_bf16x2(acc[8 * x + 4] * inv_L, acc[8 * x + 5] * inv_L),
                                    pack_bf16x2(acc[8 * x + 6] * inv_L, acc[8 * x + 7] * inv_L));
        }
    }
}

// SELF: a batch of one prefill request, planned by the kernel itself (pieces in
// shared memory); else the plan kernel's lists in the workspace.
template <int D, int NQ, bool SELF>
__global__ void __launch_bounds__(352, 1)
chunk_attn_kernel(const ChunkParams p, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_kn, const __grid_constant__ CUtensorMap tm_vn,
                  const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_v4)
{
    using C = ChunkCfg<D, NQ>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    ChunkBars *bars = reinterpret_cast<ChunkBars *>(smem + C::kBarOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        // a K or V tile is filled by the producer's issuer lanes, one arrival each
        const uint32_t issuers = (uint32_t)(128 / (p.page_size < 128 ? p.page_size : 128)) * C::kHalves;
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->q_empty, 1);
        mbar_init(&bars->tail, issuers);
        mbar_init(&bars->drain, 1);
        for (int n = 0; n < 2; ++n) {
            mbar_init(&bars->s_full[n], 1);
            mbar_init(&bars->p_full[n], 4);
            mbar_init(&bars->o_done[n], 1);
        }
        for (int s = 0; s < C::kSlots; ++s) {
            mbar_init(&bars->slot_full[s], issuers);
            mbar_init(&bars->slot_empty[s], 1);
        }
        mbar_init(&bars->stage, 1);
        mbar_init(&bars->writer_done, 1);
        bars->abort = 0;
        fence_barrier_init();
    }
    if (warp == C::kLoadWarp && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        if (D == 128 && p.out_tma)
            tma_prefetch_desc(&tm_o);
        if (D == 128 && p.page_size < 128)
            tma_prefetch_desc(&tm_v4);
        if (p.fused) {
            tma_prefetch_desc(&tm_kn);
            tma_prefetch_desc(&tm_vn);
        }
    }
    if (warp == C::kMmaWarp) {
        tmem_alloc(&bars->tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    // the set-up above touches no global memory; from here on the plan's output
    pdl_wait();
    PrefillItem *s_items = reinterpret_cast<PrefillItem *>(smem + C::kItemOff);
    if (SELF) {
        // a batch of one prefill request: this CTA computes its own run; meanwhile
        // the producer pulls the start of the request's block_table row into L2
        // (up to 32 lines, within the row), which its first lookups read next
        if (warp == C::kLoadWarp && lane * 32 < p.max_blocks)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p.block_table + lane * 32));
        if (warp == C::kWriteWarp) {
            const SelfPlanArgs a{p.query_lens, p.seq_lens, p.dev_err, p.num_tokens, p.max_blocks, p.page_size,
                                 p.group, p.num_kv_heads, p.fused, p.split_ok, p.split_clamped};
            const int n = self_plan_run<NQ>(a, s_items, lane);
            if (lane == 0) {
                bars->it_begin = 0;
                bars->it_end = n;
            }
        }
    } else if (threadIdx.x == 0) {
        // this CTA's run of pieces, from the plan's table
        bars->it_begin = p.run_first[blockIdx.x];
        bars->it_end = p.run_first[blockIdx.x + 1];
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    volatile int *abort = &bars->abort;
    const int it_begin = bars->it_begin, it_end = bars->it_end;
    const PrefillItem *items = SELF ? s_items : p.pitems;
    // first row of a request in q / out (a self-planned batch has one request)
    auto row0 = [&](int r) -> int { return SELF ? 0 : p.cu_q[r]; };

    if (warp == C::kLoadWarp) {
        // ------------------------------------------------------------ producer
        const int PB = p.page_size < 128 ? p.page_size : 128;   // rows per TMA box
        const int NB = 128 / PB;                                 // boxes per tile
        const uint32_t box_bytes = (uint32_t)PB * 128u;
        const bool v_pages = D == 128 && PB < 128;   // V tiles of the cache in page-major boxes
        uint32_t q_uses = 0, slot_it = 0, tail_uses = 0;
        for (int it = it_begin; it < it_end && !*abort; ++it) {
            const PrefillItem w = items[it];
            const int kvh = w.kvh_hp & 0xFFFF, hp = w.kvh_hp >> 16;
            const int h0 = kvh * p.group + hp * NQ;
            const int cu = row0(w.r);
            const int s_len = p.seq_lens[w.r];
            const int hist = s_len - p.query_lens[w.r];
            // tiles [0, nh) come from the cache, over keys [0, hist_end); the rest
            // (fused KV write) from the new rows
            const int nh = p.fused ? (hist + 127) / 128 : 0x7fffffff;
            const int hist_end = p.fused ? hist : s_len;
            if (q_uses > 0 && !mbar_wait(&bars->q_empty, (q_uses - 1) & 1, abort))
                break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars->q_full, NQ * C::kTileBytes);
                for (int n = 0; n < NQ; ++n)
                    for (int c = 0; c < C::kHalves; ++c)
                        tma_load_3d(smem + C::kQOff + n * C::kTileBytes + c * C::kHalfBytes, &tm_q,
                                    &bars->q_full, c * 64, h0 + n, cu + w.i0);
            }
            ++q_uses;
            const int32_t *bt_row = p.block_table + (int64_t)w.r * p.max_blocks;
            // Lane l < NB * kHalves (an issuer lane) copies box j = l % NB (rows
            // j*PB .. j*PB+PB-1 of a tile), half c = l / NB, so a tile's boxes go out
            // in one warp instruction rather than one lane's serial loop (16 boxes a
            // tile at page 16). Every issuer lane arrives once on the tile's barrier
            // (the barrier counts NB * kHalves arrivals): with the expected bytes of
            // its own copy right before issuing it, or without bytes when its box is
            // not loaded. The bytes a copy delivers are thus always announced first
            // by the lane that issues it, whatever order the lanes run in. Each issuer
            // lane holds the page of its box; the lookup for tile kt + 1 is issued
            // while tile kt's copies are set up (one tile ahead).
            const int box = lane % NB, half = lane / NB;
            const bool issuer = lane < NB * C::kHalves;
            auto lookup = [&](int kt) -> int {
                int pg = -1;
                const int key = kt * 128 + box * PB;
                if (issuer && kt < w.kt1 && kt < nh && key < hist_end)
                    pg = __ldg(bt_row + key / p.page_size);
                return pg;
            };
            int next_page = lookup(w.kt0);
            bool stop = false;
            for (int kt = w.kt0; kt < w.kt1 && !stop; ++kt) {
                const bool from_new = kt >= nh;
                const int key0 = from_new ? hist + (kt - nh) * 128 : kt * 128;
                const int key_end = from_new ? s_len : hist_end;   // keys [key0, key_end) are used
                const int page = next_page;
                next_page = lookup(kt + 1);
                const int off = (key0 + box * PB) % p.page_size;
                bool valid = false;
                if (!from_new && issuer && key0 + box * PB < key_end) {
                    valid = page >= 0 && page < p.num_pages;
                    if (!valid && half == 0)
                        set_dev_error(p.dev_err, CPSA_DEV_PAGE_OUT_OF_RANGE);
                }
                const bool tail = key0 + 128 > key_end;
                for (int kv = 0; kv < 2 && !stop; ++kv) {
                    const int slot = slot_it % C::kSlots;
                    if (slot_it >= (uint32_t)C::kSlots &&
                        !mbar_wait(&bars->slot_empty[slot], ((slot_it / C::kSlots) - 1) & 1, abort)) {
                        stop = true;
                        break;
                    }
                    uint8_t *dst = smem + C::kSlotOff + slot * C::kTileBytes;
                    const bool fix = kv == 1 && tail;
                    uint64_t *bar = fix ? &bars->tail : &bars->slot_full[slot];
                    if (from_new) {
                        // rows of tokens cu + key0 - hist .. + 127, kv head kvh: lane c loads
                        // half c (a box of new rows is always whole; rows past the tile's
                        // last key are zeroed below when the tile is a tail)
                        if (lane < C::kHalves) {
                            mbar_arrive_expect_tx(bar, C::kHalfBytes);
                            tma_load_3d(dst + lane * C::kHalfBytes, kv == 0 ? &tm_kn : &tm_vn, bar, lane * 64, kvh,
                                        cu + key0 - hist);
                        } else if (issuer) {
                            mbar_arrive(bar);
                        }
                    } else if (valid && kv == 1 && v_pages) {
                        // V below page 128: one box per page holding both column halves,
                        // [page][half][PB rows][128 B] (the half-1 lanes only arrive)
                        if (half == 0) {
                            mbar_arrive_expect_tx(bar, 2 * box_bytes);
                            tma_load_4d(dst + box * 2 * box_bytes, &tm_v4, bar, 0, off, 0,
                                        page * p.num_kv_heads + kvh);
                        } else {
                            mbar_arrive(bar);
                        }
                    } else if (valid) {
                        mbar_arrive_expect_tx(bar, box_bytes);
                        tma_load_3d(dst + half * C::kHalfBytes + box * box_bytes, kv == 0 ? &tm_k : &tm_v, bar,
                                    half * 64, off, page * p.num_kv_heads + kvh);
                    } else if (issuer) {
                        mbar_arrive(bar);
                    }
                    if (fix) {
                        // value rows >= key_end must be zero: P is zero there, but the
                        // bytes may be NaN and 0 * NaN would poison the row sums.
                        if (!mbar_wait(&bars->tail, tail_uses & 1, abort)) {
                            stop = true;
                            break;
                        }
                        ++tail_uses;
                        const int first = key_end - key0;   // 1 .. 127
                        const int nchunks = (128 - first) * 8;   // 16-byte chunks per half
                        if (v_pages && !from_new) {
                            // [page][half][PB rows][128 B]: row r, half c at
                            // (r / PB) * 2 * box_bytes + c * box_bytes + (r % PB) * 128
                            for (int x = lane; x < 2 * nchunks; x += 32) {
                                const int r = first + (x >> 4), c = (x >> 3) & 1;
                                uint4 *q = reinterpret_cast<uint4 *>(dst + (r / PB) * 2 * box_bytes + c * box_bytes +
                                                                     (r % PB) * 128);
                                q[x & 7] = make_uint4(0, 0, 0, 0);
                            }
                        } else {
                            for (int c = 0; c < C::kHalves; ++c)
                                for (int x = lane; x < nchunks; x += 32) {
                                    uint4 *row = reinterpret_cast<uint4 *>(dst + c * C::kHalfBytes + first * 128);
                                    row[x] = make_uint4(0, 0, 0, 0);
                                }
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (issuer)
                            mbar_arrive(&bars->slot_full[slot]);
                    }
                    ++slot_it;
                }
            }
            if (stop)
                break;
        }
    } else if (warp == C::kWriteWarp) {
        // ------------------------------------------------------------ cache writer
        // Independent of the attention pipeline: it reads the new rows itself,
        // one K or V tile at a time, through its own buffer and barrier.
        if (p.fused) {
            uint8_t *stage = smem + C::kStageOff;
            uint32_t stage_uses = 0;
            bool ok = true;
            for (int it = it_begin; it < it_end && ok && !*abort; ++it) {
                const PrefillItem w = items[it];
                const int kvh = w.kvh_hp & 0xFFFF, hp = w.kvh_hp >> 16;
                const int q_len = p.query_lens[w.r];
                const int hist = p.seq_lens[w.r] - q_len;
                const int kd = hp == 0 ? (hist + 127) / 128 + w.i0 / 128 : -1;
                if (kd < w.kt0 || kd >= w.kt1)
                    continue;
                const int rows = min(128, q_len - w.i0);
                const int t0 = row0(w.r) + w.i0;
                int64_t sl[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int row = lane + 32 * q;
                    sl[q] = row < rows ? __ldg(p.slot_mapping + t0 + row) : -1;
                }
                // which boxes of PB rows go whole by TMA: valid rows, slots
                // consecutive from a box start that leaves the box inside its page
                const int PB = p.page_size < 128 ? p.page_size : 128;
                const int64_t n_slots = p.num_pages * (int64_t)p.page_size;
                uint32_t okm[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int row = lane + 32 * q;
                    const int64_t sv = sl[q];
                    int64_t prev = __shfl_up_sync(0xffffffffu, sv, 1);
                    const int64_t wrap = __shfl_sync(0xffffffffu, q > 0 ? sl[q > 0 ? q - 1 : 0] : -2, 31);
                    if (lane == 0)
                        prev = wrap;
                    bool good = row < rows && sv >= 0 && sv < n_slots;
                    if (row % PB == 0)
                        good = good && (sv & (p.page_size - 1)) + PB <= p.page_size;
                    else
                        good = good && sv == prev + 1;
                    okm[q] = __ballot_sync(0xffffffffu, good);
                }
                uint32_t box_mask = 0;
                int64_t s0[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    if (j < 128 / PB) {
                        const int r0 = j * PB;
                        const int q0 = r0 >> 5;
                        bool whole;
                        if (PB >= 32) {
                            whole = true;
                            for (int q = q0; q < ((r0 + PB) >> 5); ++q)
                                whole = whole && okm[q] == 0xffffffffu;
                        } else {
                            const uint32_t m = ((1u << PB) - 1u) << (r0 & 31);
                            whole = (okm[q0] & m) == m;
                        }
                        const int64_t mine = q0 == 0 ? sl[0] : q0 == 1 ? sl[1] : q0 == 2 ? sl[2] : sl[3];
                        s0[j] = __shfl_sync(0xffffffffu, mine, r0 & 31);
                        box_mask |= (whole ? 1u : 0u) << j;
                    }
                }
                for (int kv = 0; kv < 2 && ok; ++kv) {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&bars->stage, C::kTileBytes);
                        for (int c = 0; c < C::kHalves; ++c)
                            tma_load_3d(stage + c * C::kHalfBytes, kv == 0 ? &tm_kn : &tm_vn, &bars->stage, c * 64,
                                        kvh, t0);
                    }
                    ok = __all_sync(0xffffffffu, mbar_wait_sleep(&bars->stage, stage_uses & 1u, abort));
                    if (!ok) {
                        // let the copy in flight land before the CTA can end
                        if (lane == 0) {
                            const uint64_t ts = global_timer_ns();
                            while (!mbar_try_wait(&bars->stage, stage_uses & 1u) &&
                                   global_timer_ns() - ts < 100000000ull) {
                            }
                        }
                        break;
                    }
                    ++stage_uses;
                    store_tile_rows<D>(p, kv == 0 ? &tm_k : &tm_v, stage, kv == 0 ? p.k_cache_w : p.v_cache_w, kvh,
                                       rows, sl, box_mask, s0, PB, lane, kv == 0);
                    if (lane == 0)
                        bulk_wait_group_read0();   // the TMA stores have read the buffer
                    fence_proxy_async_smem();      // and so have this warp's row copies, before the next load
                    __syncwarp();
                }
            }
            // every store has read the buffer (each job waits for that): release it
            // to the epilogue, then let the stores complete before the CTA ends
            if (lane == 0) {
                mbar_arrive(&bars->writer_done);
                bulk_wait_group0();
            }
        } else if (lane == 0) {
            mbar_arrive(&bars->writer_done);
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp walks the loop; every MMA and commit is issued by one
        // lane from an elect.sync branch. Waits are polled by all lanes and their
        // verdicts combined, so the warp stays converged.
        constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
        const uint32_t q_addr = smem_u32(smem + C::kQOff);
        const uint32_t slot_addr = smem_u32(smem + C::kSlotOff);
        uint32_t q_uses = 0, slot_it = 0, p_uses[2] = {0, 0};
        auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
            const bool ok = mbar_wait(bar, parity, abort);
            return __all_sync(0xffffffffu, ok);
        };
        auto aborted = [&]() -> bool { return __any_sync(0xffffffffu, *abort != 0); };
        auto commit = [&](uint64_t *bar) {
            if (elect_one_sync())
                umma_commit(bar);
        };
        auto issue_qk = [&](int n, int slot) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t koff = (kk >> 2) * C::kHalfBytes + (kk & 3) * 32;
                const uint64_t a = smem_desc_sw128(q_addr + n * C::kTileBytes + koff, 0, 1024);
                const uint64_t b = smem_desc_sw128(slot_addr + slot * C::kTileBytes + koff, 0, 1024);
                if (elect_one_sync())
                    umma_ss(tmem + C::s_col(n), a, b, idesc_qk, kk > 0);
            }
        };
        // V below page 128 (cache tiles) lands page-major, [page][half][P rows][128 B]:
        // keys 16 kk .. 16 kk + 15 start at page 16 kk / P, row 16 kk % P; the
        // column halves are P * 128 bytes apart, 8-key groups 1024 bytes (two pages
        // at page 8). Otherwise [half][128 rows][128 B].
        const int pg = p.page_size < 128 ? p.page_size : 128;
        const int lg_pg = __ffs(pg) - 1;
        const bool v_pages = D == 128 && pg < 128;
        auto issue_pv = [&](int n, int slot, bool acc, bool pm) {
#pragma unroll
            for (int kk = 0; kk < 128 / 16; ++kk) {
                const int r0 = kk * 16;
                const uint32_t off = pm ? (uint32_t)(((r0 >> lg_pg) << (lg_pg + 8)) + (r0 & (pg - 1)) * 128)
                                        : (uint32_t)(r0 * 128);
                const uint64_t b = smem_desc_sw128(slot_addr + slot * C::kTileBytes + off,
                                                   pm ? (uint32_t)pg * 128u : (uint32_t)C::kHalfBytes,
                                                   pm && pg < 16 ? (uint32_t)pg * 256u : 1024u);
                if (elect_one_sync())
                    umma_ts(tmem + C::o_col(n), tmem + C::s_col(n) + kk * 8, b, idesc_pv, (acc || kk > 0));
            }
        };
        auto wait_slot = [&](int &slot) -> bool {
            slot = slot_it % C::kSlots;
            const bool ok = wait(&bars->slot_full[slot], (slot_it / C::kSlots) & 1);
            ++slot_it;
            tc_fence_after_sync();
            return ok;
        };
        for (int it = it_begin; it < it_end && !aborted(); ++it) {
            const PrefillItem w = items[it];
            const int n = w.kt1 - w.kt0;
            // tiles from nh on hold the chunk's own keys, loaded from k/v (fused KV write)
            const int nh = v_pages && p.fused ? (p.seq_lens[w.r] - p.query_lens[w.r] + 127) / 128 : 0x7fffffff;
            if (!wait(&bars->q_full, q_uses & 1))
                break;
            ++q_uses;
            tc_fence_after_sync();
            int sK, sV;
            if (!wait_slot(sK))
                break;
            for (int qn = 0; qn < NQ; ++qn) {
                issue_qk(qn, sK);
                commit(&bars->s_full[qn]);
            }
            commit(&bars->slot_empty[sK]);
            if (n == 1)
                commit(&bars->q_empty);
            bool ok = true;
            for (int t = 0; t < n && ok; ++t) {
                if (!(ok = wait_slot(sV)))
                    break;
                if (!(ok = wait(&bars->p_full[0], p_uses[0] & 1)))
                    break;
                ++p_uses[0];
                tc_fence_after_sync();
                const bool pm = v_pages && w.kt0 + t < nh;
                issue_pv(0, sV, t > 0, pm);
                commit(&bars->o_done[0]);
                const bool more = t + 1 < n;
                if (more) {
                    if (!(ok = wait_slot(sK)))
                        break;
                    issue_qk(0, sK);
                    commit(&bars->s_full[0]);
                }
                if (NQ == 2) {
                    if (!(ok = wait(&bars->p_full[1], p_uses[1] & 1)))
                        break;
                    ++p_uses[1];
                    tc_fence_after_sync();
                    issue_pv(1, sV, t > 0, pm);
                    commit(&bars->o_done[1]);
                }
                commit(&bars->slot_empty[sV]);
                if (more) {
                    if (NQ == 2) {
                        issue_qk(1, sK);
                        commit(&bars->s_full[1]);
                    }
                    commit(&bars->slot_empty[sK]);
                    if (t + 2 == n)
                        commit(&bars->q_empty);
                }
            }
            if (!ok)
                break;
        }
        if (aborted()) {
            // let every MMA issued so far finish before TMEM is released
            commit(&bars->drain);
            if (lane == 0) {
                uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(&bars->drain, 0) && global_timer_ns() - t0 < 100000000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp / 4 < NQ) {
        // ------------------------------------------------------------ softmax
        const int wg = warp / 4;
        const int sub = warp & 3;
        const int row = sub * 32 + lane;
        const uint32_t lane_base = (uint32_t)(sub * 32) << 16;
        const uint32_t tS = tmem + lane_base + C::s_col(wg);
        const uint32_t tO = tmem + lane_base + C::o_col(wg);
        const float sl2 = p.scale_log2;
        uint32_t s_uses = 0, o_base = 0;
        for (int it = it_begin; it < it_end && !*abort; ++it) {
            const PrefillItem w = items[it];
            const int kvh = w.kvh_hp & 0xFFFF, hp = w.kvh_hp >> 16;
            const int h = kvh * p.group + hp * NQ + wg;
            const int q_len = p.query_lens[w.r];
            const int s_len = p.seq_lens[w.r];
            const int hist = s_len - q_len;
            const int i = w.i0 + row;
            const int limit = min(hist + i, s_len - 1);   // last visible key of this row
            // with the KV write fused, tiles from nh on hold the chunk's own keys
            // from key hist on, and the cache tiles before them end at hist
            const int nh = p.fused ? (hist + 127) / 128 : 0x7fffffff;
            const int limit_hist = p.fused ? hist - 1 : limit;
            const int n = w.kt1 - w.kt0;
            float m_use = -INFINITY, l = 0.f;
            bool ok = true;
            for (int t = 0; t < n; ++t) {
                const int kt = w.kt0 + t;
                const bool from_new = kt >= nh;
                const int key0 = from_new ? hist + (kt - nh) * 128 : kt * 128;
                const int lim = from_new ? limit : limit_hist;
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[wg], s_uses & 1, abort))))
                    break;
                ++s_uses;
                tc_fence_after_sync();
                // the S row straight from TMEM: four loads, one wait
                uint32_t sr[4][32];
                float rm[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32_max(tS + c * 32, sr[c], rm[c]);
                tmem_wait_ld();
#define SV(x) __uint_as_float(sr[(x) >> 5][(x) & 31])
                // causal / tail mask: only tiles that reach past some row's last key
                const bool masked = __any_sync(0xffffffffu, key0 + 127 > lim);
                float mx = fmaxf(fmaxf(rm[0], rm[1]), fmaxf(rm[2], rm[3]));
                if (masked) {
#pragma unroll
                    for (int x = 0; x < 128; ++x)
                        if (key0 + x > lim) sr[x >> 5][x & 31] = 0xff800000u;   // -inf
                    // row max as 4 independent fmax3 chains joined at the end (short latency)
                    float mc[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) mc[c] = fmaxf(SV(c), SV(c + 4));
#pragma unroll
                    for (int x = 8; x < 128; x += 8)
#pragma unroll
                        for (int c = 0; c < 4; ++c) mc[c] = fmax3(mc[c], SV(x + c), SV(x + 4 + c));
                    mx = fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3]));
                }
                const float m_tile = mx * sl2;
                const bool need = m_tile > m_use + 8.f;
                float alpha = 1.f;
                if (need) {
                    alpha = ex2_approx(m_use - m_tile);   // m_use = -inf gives 0
                    l *= alpha;
                    m_use = m_tile;
                }
                const float mref = m_use == -INFINITY ? 0.f : m_use;
                const uint64_t sl2x2 = f2_pack(sl2, sl2);
                const uint64_t nref2 = f2_pack(-mref, -mref);
                uint64_t sum2 = f2_pack(0.f, 0.f);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t pk[32];
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        // exponent of the pair (s * scale * log2e - m) in one packed FMA
                        const uint64_t e2 = f2_fma(f2_pack(SV(64 * hh + 2 * x), SV(64 * hh + 2 * x + 1)), sl2x2, nref2);
                        float a, b;
                        if (!masked && (x & 7) < kFmaExpPairsPer8) {
                            f2_unpack(e2, a, b);
                            f2_unpack(exp2_poly_x2(f2_pack(fmaxf(a, -125.f), fmaxf(b, -125.f))), a, b);
                        } else {
                            f2_unpack(e2, a, b);
                            a = ex2_approx(a);
                            b = ex2_approx(b);
                        }
                        const uint64_t p2 = f2_pack(a, b);
                        sum2 = f2_add(sum2, p2);
                        pk[x] = pack_bf16x2(a, b);
                    }
                    tmem_st32(tS + 32 * hh, pk);
                }
#undef SV
                {
                    float s0, s1;
                    f2_unpack(sum2, s0, s1);
                    l += s0 + s1;
                }
                tmem_wait_st();
                if (__any_sync(0xffffffffu, need) && t > 0) {
                    // O holds the sum through tile t-1: wait for that P.V, then rescale
                    if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_done[wg], (o_base + t - 1) & 1, abort))))
                        break;
                    tc_fence_after_sync();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32(tO + c * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int x = 0; x < 32; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * alpha);
                        tmem_st32(tO + c * 32, r);
                    }
                    tmem_wait_st();
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&bars->p_full[wg]);
            }
            if (!ok)
                break;
            if (!__all_sync(0xffffffffu, mbar_wait(&bars->o_done[wg], (o_base + n - 1) & 1, abort)))
                break;
            o_base += n;
            tc_fence_after_sync();
            const bool valid_row = i < q_len;
            const int64_t t_row = (int64_t)row0(w.r) + i;
            const int npieces = w.piece_np >> 16;
            if (npieces > 1) {
                // A piece of a split unit. Every warp (32 rows) decides on its own:
                // at the end of its CTA's run, if every other piece has left its
                // partial, it merges them with its own O at once (the usual case:
                // its partner pieces ran at the start of the next CTAs' runs);
                // else it leaves its partial and counts itself in, and the piece whose
                // count completes the set merges. No warp waits for another piece.
                // Partials are O / l in bf16 (m and l in fp32 beside them), column-major
                // per (piece, head): the 8 columns 8j .. 8j + 7 of row `row` as one
                // 16-byte unit at ((piece * NQ + wg) * D/8 + j) * 128 + row, so a warp's
                // accesses are 512 contiguous bytes. The unit's partial rows keep
                // the fp32 row pitch of the workspace (decode partials share it).
                const int piece = w.piece_np & 0xFFFF;
                unsigned long long *cnt = p.flags + ((int64_t)w.aux * NQ + wg) * 4 + sub;
                uint4 *ph = reinterpret_cast<uint4 *>(p.part_o) + (int64_t)w.pbase * (D / 4);
                float2 *pml = reinterpret_cast<float2 *>(p.part_ml) + w.pbase;
                // lane 0 reads the counter now: at the run's last item to see whether the
                // other pieces are all in (acquire: their partials are read next),
                // otherwise only as the guess for counting in (relaxed: an acquire
                // would hold this lane's partial stores back until it returns)
                unsigned long long cur = 0;
                int seen = 0;
                if (lane == 0) {
                    if (it + 1 == it_end) {
                        cur = ld_acquire_gpu_u64(cnt);
                        seen = epoch_count(cur, p.epoch);
                    } else {
                        cur = ld_relaxed_gpu_u64(cnt);
                    }
                }
                seen = __shfl_sync(0xffffffffu, seen, 0);
                bool merge = seen == npieces - 1;
                if (!merge) {
                    const float inv_own = l > 0.f ? 1.f / l : 0.f;
                    uint4 *dst = ph + (int64_t)(piece * NQ + wg) * (D / 8) * 128 + row;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32(tO + c * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int x = 0; x < 4; ++x)
                            dst[(c * 4 + x) * 128] =
                                make_uint4(pack_bf16x2(__uint_as_float(r[8 * x + 0]) * inv_own, __uint_as_float(r[8 * x + 1]) * inv_own),
                                           pack_bf16x2(__uint_as_float(r[8 * x + 2]) * inv_own, __uint_as_float(r[8 * x + 3]) * inv_own),
                                           pack_bf16x2(__uint_as_float(r[8 * x + 4]) * inv_own, __uint_as_float(r[8 * x + 5]) * inv_own),
                                           pack_bf16x2(__uint_as_float(r[8 * x + 6]) * inv_own, __uint_as_float(r[8 * x + 7]) * inv_own));
                    }
                    pml[(piece * NQ + wg) * 128 + row] = make_float2(m_use, l);
                    __syncwarp();
                    if (lane == 0) {
                        fence_acq_rel_gpu();   // this warp's partial, then the count
                        seen = epoch_arrive(cnt, p.epoch, cur, p.dev_err);
                        fence_acq_rel_gpu();   // the count, then the other partials
                    }
                    seen = __shfl_sync(0xffffffffu, seen, 0);
                    merge = seen == npieces - 1;
                }
                if (merge) {
                    const int64_t out_off = (t_row * p.num_q_heads + h) * D;
                    if (npieces - 1 <= kMergeMaxOthers) {
                        // at the run's last item the Q and K/V buffers are free once the
                        // other head's last P.V is done: the merge stages through them
                        bool staged = false;
                        if (D == 128 && it + 1 == it_end)
                            staged = NQ == 1 || __all_sync(0xffffffffu, mbar_wait(&bars->o_done[NQ - 1 - wg],
                                                                                  (o_base - 1) & 1, abort));
                        // the merged rows through the writer's buffer once the writer is done with it
                        const bool ostaged = staged && p.out_tma &&
                                             (!p.fused || __all_sync(0xffffffffu, mbar_wait(&bars->writer_done, 0, abort)));
                        merge_split_row<D, NQ>(p, tO, pml, ph, piece, npieces, wg, row, lane, m_use, l, valid_row,
                                               out_off,
                                               staged ? reinterpret_cast<uint4 *>(smem + (wg * 4 + sub) * kMergeStageBytes)
                                                      : nullptr,
                                               ostaged ? smem + C::kStageOff + (wg * 4 + sub) * 4096 : nullptr, &tm_o, h,
                                               (int)(t_row - lane));
                    } else {
                        merge_split_row_any<D, NQ>(p, tO, pml, ph, piece, npieces, wg, row, m_use, l, valid_row,
                                                   out_off);
                    }
                    // Every other piece has counted in, so no one else touches the
                    // counter in this call: the merging warp clears it. A later call
                    // then finds it clear even under the same epoch (a call captured
                    // in a CUDA graph replays its epoch).
                    if (lane == 0)
                        *reinterpret_cast<volatile unsigned long long *>(cnt) = 0ull;
                }
            } else if constexpr (!SELF && D == 128) {
                // A whole unit of a planned batch. Without the KV write (whose cache
                // writer holds the buffer) each warp stages its 32 rows, 64 columns
                // at a time, in its own 4 KB of the writer's buffer and a TMA store
                // writes them out, so the warp moves on to the next unit while the
                // rows go to memory; a warp with rows past the request's end (the
                // last query tile), or any warp of a call with the KV write, stores
                // its valid rows directly. (Planned batches hold many units per
                // run; the self-planned kernel, with few, stores directly: staging
                // measured slower there.)
                const float inv_l = l > 0.f ? 1.f / l : 0.f;
                // with the KV write, once the cache writer has released its buffer
                const bool writer_idle =
                    !p.fused || __shfl_sync(0xffffffffu, lane == 0 && mbar_test_wait(&bars->writer_done, 0), 0);
                const bool staged = p.out_tma && writer_idle && __all_sync(0xffffffffu, valid_row);
                uint8_t *stg = smem + C::kStageOff + (wg * 4 + sub) * 4096;
#pragma unroll
                for (int c2 = 0; c2 < D / 64; ++c2) {
                    // 64 columns into registers first: the wait for the previous
                    // store's read (the other half's, just issued) overlaps the TMEM loads
                    uint4 v[2][4];
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        uint32_t r[32];
                        tmem_ld32(tO + (2 * c2 + cc) * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int x = 0; x < 4; ++x)
                            v[cc][x] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * x + 0]) * inv_l, __uint_as_float(r[8 * x + 1]) * inv_l),
                                                  pack_bf16x2(__uint_as_float(r[8 * x + 2]) * inv_l, __uint_as_float(r[8 * x + 3]) * inv_l),
                                                  pack_bf16x2(__uint_as_float(r[8 * x + 4]) * inv_l, __uint_as_float(r[8 * x + 5]) * inv_l),
                                                  pack_bf16x2(__uint_as_float(r[8 * x + 6]) * inv_l, __uint_as_float(r[8 * x + 7]) * inv_l));
                    }
                    if (staged) {
                        if (lane == 0)
                            bulk_wait_group_read0();   // the warp's previous store has read the buffer
                        __syncwarp();
                        // row `lane` at lane * 128 bytes, 16-byte chunk j at (j ^ (lane & 7)):
                        // the map's 128-byte swizzle
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                            for (int x = 0; x < 4; ++x)
                                *reinterpret_cast<uint4 *>(stg + lane * 128 + (((cc * 4 + x) ^ (lane & 7)) << 4)) = v[cc][x];
                    } else if (valid_row) {
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) {
                            uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) +
                                                                   (t_row * p.num_q_heads + h) * D + (2 * c2 + cc) * 32);
#pragma unroll
                            for (int x = 0; x < 4; ++x)
                                dst[x] = v[cc][x];
                        }
                    }
                    if (staged) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_3d(&tm_o, stg, c2 * 64, h, (int)(t_row - lane));
                            bulk_commit_group();
                        }
                    }
                }
            } else if (SELF && D == 128 && p.out_tma &&
                       (!p.fused || __shfl_sync(0xffffffffu, lane == 0 && mbar_test_wait(&bars->writer_done, 0), 0))) {
                store_unit_rows_staged<D>(tO, l, valid_row, smem + C::kStageOff + (wg * 4 + sub) * 4096, &tm_o,
                                          reinterpret_cast<__nv_bfloat16 *>(p.out), t_row, h, p.num_q_heads, lane);
            } else {
                const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tO + c * 32, r);
                    tmem_wait_ld();
                    if (valid_row) {
                        uint4 *dst = reinterpret_cast<uint4 *>(
                            reinterpret_cast<__nv_bfloat16 *>(p.out) + (t_row * p.num_q_heads + h) * D + c * 32);
#pragma unroll
                        for (int x = 0; x < 4; ++x)
                            dst[x] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * x + 0]) * inv_l, __uint_as_float(r[8 * x + 1]) * inv_l),
                                                pack_bf16x2(__uint_as_float(r[8 * x + 2]) * inv_l, __uint_as_float(r[8 * x + 3]) * inv_l),
                                                pack_bf16x2(__uint_as_float(r[8 * x + 4]) * inv_l, __uint_as_float(r[8 * x + 5]) * inv_l),
                                                pack_bf16x2(__uint_as_float(r[8 * x + 6]) * inv_l, __uint_as_float(r[8 * x + 7]) * inv_l));
                    }
                }
            }
        }
    }

    // the softmax warps' output stores are complete before the CTA ends
    if (D == 128 && warp / 4 < NQ && lane == 0 && p.out_tma)
        bulk_wait_group0();
    if (threadIdx.x == 0 && bars->abort)
        set_dev_error(p.dev_err, CPSA_DEV_WAIT_TIMEOUT);
    // The next kernels are released only as CTAs finish: launched at the start
    // they would wait beside this CTA's warps for its whole run (measured slower).
    pdl_trigger();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, int NQ>
cudaError_t launch_chunk_t(const ChunkParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                           const CUtensorMap &tv, const CUtensorMap &tkn, const CUtensorMap &tvn,
                           const CUtensorMap &to, const CUtensorMap &tv4, int grid, cudaStream_t s, bool early)
{
    using C = ChunkCfg<D, NQ>;
    static std::atomic<uint64_t> done_self{0}, done_plan{0};
    auto k = p.self_plan ? chunk_attn_kernel<D, NQ, true> : chunk_attn_kernel<D, NQ, false>;
    return launch_with_smem(p.self_plan ? done_self : done_plan, reinterpret_cast<const void *>(k), C::kSmemBytes,
                            [&] {
                                return launch_pdl(early, k, dim3(grid), dim3(C::kThreads), C::kSmemBytes, s, p, tq,
                                                  tk, tv, tkn, tvn, to, tv4);
                            });
}

}  // namespace

cudaError_t launch_chunk_attn(const ChunkParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                              const CUtensorMap &tv, const CUtensorMap &tkn, const CUtensorMap &tvn,
                              const CUtensorMap &to, const CUtensorMap &tv4, int head_dim, int nq, int grid,
                              cudaStream_t s, bool early)
{
    if (head_dim == 128)
        return nq == 2 ? launch_chunk_t<128, 2>(p, tq, tk, tv, tkn, tvn, to, tv4, grid, s, early)
                       : launch_chunk_t<128, 1>(p, tq, tk, tv, tkn, tvn, to, tv4, grid, s, early);
    return nq == 2 ? launch_chunk_t<64, 2>(p, tq, tk, tv, tkn, tvn, to, tv4, grid, s, early)
                   : launch_chunk_t<64, 1>(p, tq, tk, tv, tkn, tvn, to, tv4, grid, s, early);
}

}  // namespace cpsa
