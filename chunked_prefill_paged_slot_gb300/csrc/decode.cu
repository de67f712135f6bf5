// decode.cu -- split-KV attention of decode rows (query_len == 1) over the paged
// cache. HBM-bound: every key and value of the row's context is read once per
// kv head, for all q heads of that kv head at once (GQA grouping).
//
// What it computes ("vLLM Chunked-Prefills" article, section 3.1: decode rows
// ride in the same step as the prefill chunk, one token each; attention per
// section 3.2.1): for the single new token of request r and the q heads
// kvh*G .. kvh*G+G-1, softmax(scale * q K^T) V over keys [key0, key1) of the
// row's context (a whole context, or one split of it).
//
// CTA layout (160 threads, persistent over decode items):
//   last warp  producer: 64-key stages of K and V through TMA, one box per
//              page-head block (or per 64 rows of a larger page) that covers
//              both 64-column halves of head_dim (a 4-D view: columns, rows,
//              halves, page-head blocks), 128-byte swizzled; the stage holds
//              [block][half][rows][128 B].
//   consumers  one or two groups of 4 warps; groups take alternate stages and
//              inside a group warp w takes keys [16w, 16w + 16) of the stage:
//              S = q K^T and O += P V with mma.sync m16n8k16
//              (the G <= 16 q heads are the M rows), online softmax in fp32
//              (base-2 exponent), partial state per warp. A stage is refilled
//              once its group's four warps are done with it.
// At the end of an item the four warps merge (max, sum, O) through shared
// memory and write the bf16 row, or an fp32 partial when the row is split.
// With the KV write fused, the row's own key (the last of its context) is not
// in the cache yet: the producer lands the stage holding it, overwrites that row
// in shared memory with the new K and V rows, stores the same bytes to the
// cache slot slot_mapping names, and only then releases the stage.
#include "common.cuh"
#include "kernels.cuh"
#include "plan.cuh"

namespace cpsa {

namespace {

constexpr int kKC = kDecodeChunk;   // keys per stage
constexpr int kLookahead = 4;       // stages of block_table lookups kept in flight

template <int D, bool HI>
struct DecCfg {
    // HI: up to 16 q heads per kv head (both halves of the mma rows); one group
    // of 4 consumer warps. Otherwise two groups take alternate stages.
    static constexpr int kGroups = HI ? 1 : 2;
    static constexpr int kConsumers = 4 * kGroups;
    static constexpr int kHalves = D / 64;
    static constexpr int kRowBytes = D * 2;
    static constexpr int kTileBytes = kKC * kRowBytes;        // K or V of one stage
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kGroupRows = HI ? kMaxGroup : 8;      // q heads per kv head, upper bound
    static constexpr int kStages = D == 128 ? 5 : 10;
    static constexpr int kMergeOff = kStages * kStageBytes;
    static constexpr int kMergeBytes = kConsumers * kGroupRows * (D + 2) * 4;
    static constexpr int kBarOff = kMergeOff + kMergeBytes;
    static constexpr int kSmemBytes = kBarOff + 256 + 1024;
    static constexpr int kThreads = 32 * (kConsumers + 1);
};

struct DecBars {
    uint64_t full[10], empty[10];
    uint64_t patch;   // fused KV write: copies of the stage that gets the new row
    int abort;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of the 128-byte half-row (row, half) in a stage tile laid out as
// [block of 2^lg rows][64-column half][row in block][128 B]; blocks are >= 8 rows.
template <int D>
__device__ __forceinline__ uint32_t half_row_off(int row, int half, int lg)
{
    const int blk = row >> lg, r = row & ((1 << lg) - 1);
    return ((uint32_t)(blk * (D / 64) + half) << (lg + 7)) + ((uint32_t)r << 7);
}

// Byte address of element (row, col) of such a tile, 128-byte swizzled: the
// 16-byte chunk c of a row sits at c ^ (row % 8) inside its half-row.
template <int D>
__device__ __forceinline__ uint32_t swz_addr(uint32_t base, int row, int col, int lg)
{
    const int ch = (col & 63) >> 3;
    return base + half_row_off<D>(row, col >> 6, lg) + ((ch ^ (row & 7)) << 4) + (col & 7) * 2;
}

template <int D, bool HI>
__global__ void __launch_bounds__(DecCfg<D, HI>::kThreads, 1)
decode_attn_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v)
{
    using C = DecCfg<D, HI>;
    constexpr int GR = C::kGroupRows;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    DecBars *bars = reinterpret_cast<DecBars *>(smem + C::kBarOff);
    float *merge = reinterpret_cast<float *>(smem + C::kMergeOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 4);
        }
        mbar_init(&bars->patch, 1);
        bars->abort = 0;
        fence_barrier_init();
    }
    // set-up above touches no global memory: from here on the plan's output
    pdl_trigger();
    pdl_wait();
    const int n_items = p.counts[kCntDecode];
    __syncthreads();
    volatile int *abort = &bars->abort;

    if (warp == C::kConsumers) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
        }
        const int PB = p.page_size < kKC ? p.page_size : kKC;
        const int NB = kKC / PB;
        const int lg = 31 - __clz(PB);
        const uint32_t box_bytes = (uint32_t)PB * C::kRowBytes;
        uint32_t g = 0, patch_uses = 0;
        bool stop = false;
        for (int it = blockIdx.x; it < n_items && !stop && !*abort; it += gridDim.x) {
            const DecodeItem w = p.ditems[it];
            const int32_t *bt_row = p.block_table + (int64_t)w.r * p.max_blocks;
            // the row's own key, when this item's range ends with it and the KV write is fused
            const int knew = (p.fused && w.key1 == p.seq_lens[w.r]) ? w.key1 - 1 : -1;
            // page numbers of the next kLookahead stages stay in flight in registers
            // (lane j < NB holds box j of a stage), so the block_table latency is
            // paid once per item rather than once per stage
            auto lookup = [&](int c) -> int {
                const int key = c + lane * PB;
                return (lane < NB && key < w.key1) ? __ldg(bt_row + key / p.page_size) : -1;
            };
            int pg[kLookahead];
#pragma unroll
            for (int k = 0; k < kLookahead; ++k) pg[k] = lookup(w.key0 + k * kKC);
            for (int c0 = w.key0; c0 < w.key1; c0 += kKC, ++g) {
                const int page = pg[0];
#pragma unroll
                for (int k = 0; k + 1 < kLookahead; ++k) pg[k] = pg[k + 1];
                pg[kLookahead - 1] = lookup(c0 + kLookahead * kKC);
                const int stage = g % C::kStages;
                if (g >= (uint32_t)C::kStages &&
                    !mbar_wait(&bars->empty[stage], ((g / C::kStages) - 1) & 1, abort)) {
                    stop = true;
                    break;
                }
                const int off = (c0 + lane * PB) % p.page_size;
                bool valid = false;
                if (lane < NB && c0 + lane * PB < w.key1) {
                    valid = page >= 0 && page < p.num_pages;
                    if (!valid)
                        set_dev_error(p.dev_err, CPSA_DEV_PAGE_OUT_OF_RANGE);
                }
                const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
                const uint32_t bytes = (uint32_t)__popc(vmask) * box_bytes * 2;
                uint8_t *kdst = smem + stage * C::kStageBytes;
                uint8_t *vdst = kdst + C::kTileBytes;
                const bool patch = knew >= c0 && knew < c0 + kKC;
                uint64_t *bar = patch ? &bars->patch : &bars->full[stage];
                if (lane == 0)
                    mbar_arrive_expect_tx(bar, bytes);
                for (int j = 0; j < NB; ++j) {
                    const int pj = __shfl_sync(0xffffffffu, page, j);
                    const int oj = __shfl_sync(0xffffffffu, off, j);
                    if (lane == 0 && ((vmask >> j) & 1u)) {
                        // rows [oj, oj + PB) of page-head block (pj, kvh), both halves in one box
                        const int z = pj * p.num_kv_heads + w.kvh;
                        if (C::kHalves == 2) {
                            tma_load_4d(kdst + j * box_bytes, &tm_k, bar, 0, oj, 0, z);
                            tma_load_4d(vdst + j * box_bytes, &tm_v, bar, 0, oj, 0, z);
                        } else {
                            tma_load_3d(kdst + j * box_bytes, &tm_k, bar, 0, oj, z);
                            tma_load_3d(vdst + j * box_bytes, &tm_v, bar, 0, oj, z);
                        }
                    }
                }
                if (patch) {
                    if (!mbar_wait(&bars->patch, patch_uses & 1u, abort)) {
                        stop = true;
                        break;
                    }
                    ++patch_uses;
                    // lanes 0..D/8-1: 16-byte chunks of the K row; lanes 16..16+D/8-1: of the V row
                    const int which = lane >> 4, ch = lane & 15;
                    if (ch < D / 8) {
                        const int rr = knew - c0;
                        const int64_t src = ((int64_t)w.t * p.num_kv_heads + w.kvh) * (D / 8) + ch;
                        const uint4 val = __ldg(reinterpret_cast<const uint4 *>(which ? p.v_new : p.k_new) + src);
                        uint8_t *tile = which ? vdst : kdst;
                        *reinterpret_cast<uint4 *>(tile + half_row_off<D>(rr, ch >> 3, lg) +
                                                   (((ch & 7) ^ (rr & 7)) << 4)) = val;
                        const int64_t slot = __ldg(p.slot_mapping + w.t);
                        if (slot >= 0) {
                            if (slot < p.num_pages * (int64_t)p.page_size) {
                                const int lg_p = __ffs(p.page_size) - 1;   // page_size is a power of two
                                const int64_t pg = slot >> lg_p, po = slot & (p.page_size - 1);
                                reinterpret_cast<uint4 *>(which ? p.v_cache_w : p.k_cache_w)
                                    [((pg * p.num_kv_heads + w.kvh) * p.page_size + po) * (D / 8) + ch] = val;
                            } else if (lane == 0) {
                                set_dev_error(p.dev_err, CPSA_DEV_SLOT_OUT_OF_RANGE);
                            }
                        }
                    }
                    fence_proxy_async_smem();   // the patch before later copies into this stage
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&bars->full[stage]);
                }
            }
        }
        return;   // the producer takes no part in the consumers' named barriers
    }

    // ---------------------------------------------------------------- consumers
    // Thread layout of mma.sync m16n8k16: A/C rows lane/4 and lane/4 + 8 (the
    // second only when HI, i.e. more than 8 q heads per kv head).
    constexpr int R = HI ? 2 : 1;
    const float sl2 = p.scale_log2;
    const int qrow = lane >> 2;
    const int qcol = (lane & 3) * 2;     // column pair within an 8-wide tile
    const int group = warp >> 2;
    const int lg = 31 - __clz(p.page_size < kKC ? p.page_size : kKC);   // log2 rows per block
    uint32_t g = 0;
    // every consumer warp walks every item (no early exit on abort: the named
    // barriers below need all four; a failed wait returns at once instead)
    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const DecodeItem w = p.ditems[it];
        const int nch = (w.key1 - w.key0 + kKC - 1) / kKC;
        // q fragments (rows >= G are zero)
        uint32_t qa[D / 16][4];
        {
            const uint32_t *qsrc = reinterpret_cast<const uint32_t *>(
                reinterpret_cast<const __nv_bfloat16 *>(p.q) + ((int64_t)w.t * p.num_q_heads + w.kvh * G) * D);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int row = qrow + 8 * rr;
                    const bool live = (rr == 0 || HI) && row < G;
                    qa[kk][rr] = live ? __ldg(qsrc + (row * D + kk * 16 + qcol) / 2) : 0u;
                    qa[kk][2 + rr] = live ? __ldg(qsrc + (row * D + kk * 16 + 8 + qcol) / 2) : 0u;
                }
            }
        }
        float m_run[R], l_run[R];
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            m_run[rr] = -INFINITY;
            l_run[rr] = 0.f;
        }
        float o[D / 8][4];
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

        for (int j = 0; j < nch; ++j) {
            const uint32_t gg = g + j;
            if ((int)(gg % C::kGroups) != group)
                continue;
            const int stage = gg % C::kStages;
            if (!mbar_wait(&bars->full[stage], (gg / C::kStages) & 1, abort))
                break;
            const int c0 = w.key0 + j * kKC;
            const int kb0 = (warp & 3) * 16;               // this warp's keys in the stage
            const int nv = min(16, w.key1 - c0 - kb0);     // valid keys of this warp (may be <= 0)
            uint8_t *kst = smem + stage * C::kStageBytes;
            uint8_t *vst = kst + C::kTileBytes;
            if (nv < 16) {
                // value rows past the range may hold anything (NaN included): zero ours
                // (whole 128-byte half-rows, so the swizzle does not matter)
                const int first = kb0 + max(nv, 0);
                const int nchunks = (kb0 + 16 - first) * C::kHalves * 8;
                for (int x = lane; x < nchunks; x += 32) {
                    const int row = first + x / (C::kHalves * 8);
                    const int half = (x >> 3) % C::kHalves;
                    *reinterpret_cast<uint4 *>(vst + half_row_off<D>(row, half, lg) + (x & 7) * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            const uint32_t kb = smem_u32(kst), vb = smem_u32(vst);
            const int mat = lane >> 3, mrow = lane & 7;
            // S = q K^T : 2 n-tiles of 8 keys
            float s[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t b0, b1, b2, b3;
                const int key = kb0 + mrow + (mat >> 1) * 8;
                const int col = kk * 16 + (mat & 1) * 8;
                ldsm_x4(swz_addr<D>(kb, key, col, lg), b0, b1, b2, b3);
                mma_bf16(s[0], qa[kk], b0, b1);
                mma_bf16(s[1], qa[kk], b2, b3);
            }
            // mask and online softmax per row (C fragment: [2rr], [2rr+1] of row qrow + 8rr)
            uint32_t pa[4];
            pa[0] = pa[1] = pa[2] = pa[3] = 0u;
#pragma unroll
            for (int rr = 0; rr < R; ++rr) {
                float mx = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        if (nt * 8 + qcol + e >= nv) s[nt][2 * rr + e] = -INFINITY;
                        mx = fmaxf(mx, s[nt][2 * rr + e]);
                    }
                }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float m_new = fmaxf(m_run[rr], mx * sl2);
                // m_run = -inf gives 0; an all-masked quarter (m_new = m_run = -inf) keeps 1
                const float alpha = m_new == m_run[rr] ? 1.f : ex2_approx(m_run[rr] - m_new);
                m_run[rr] = m_new;
                const float mref = m_new == -INFINITY ? 0.f : m_new;
                float psum = 0.f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const float p0 = ex2_approx(fmaf(s[nt][2 * rr], sl2, -mref));
                    const float p1 = ex2_approx(fmaf(s[nt][2 * rr + 1], sl2, -mref));
                    psum += p0 + p1;
                    // A fragment of P: a[rr] keys 0-7, a[2+rr] keys 8-15
                    pa[nt * 2 + rr] = pack_bf16x2(p0, p1);
                }
                l_run[rr] = l_run[rr] * alpha + psum;
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt) {
                    o[nt][2 * rr] *= alpha;
                    o[nt][2 * rr + 1] *= alpha;
                }
            }
            // O += P V : A = P (16 keys as K), B = V rows via transposed ldmatrix
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
                uint32_t b0, b1, b2, b3;
                const int key = kb0 + mrow + (mat & 1) * 8;
                const int col = np * 16 + (mat >> 1) * 8;
                ldsm_x4_t(swz_addr<D>(vb, key, col, lg), b0, b1, b2, b3);
                mma_bf16(o[2 * np], pa, b0, b1);
                mma_bf16(o[2 * np + 1], pa, b2, b3);
            }
            if (nv < 16)
                fence_proxy_async_smem();   // our zeroing writes before the next copy into this stage
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars->empty[stage]);
        }
        g += nch;
        // merge the four warps' states: max, sum, O
        float *mm = merge;                                   // [warps][GR]
        float *ll = merge + C::kConsumers * GR;              // [warps][GR]
        float *oo = merge + 2 * C::kConsumers * GR;          // [warps][GR][D]
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            float lq = l_run[rr];
            lq += __shfl_xor_sync(0xffffffffu, lq, 1);
            lq += __shfl_xor_sync(0xffffffffu, lq, 2);
            const int row = qrow + 8 * rr;
            if (row < G) {
                if ((lane & 3) == 0) {
                    mm[warp * GR + row] = m_run[rr];
                    ll[warp * GR + row] = lq;
                }
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt) {
                    oo[(warp * GR + row) * D + nt * 8 + qcol] = o[nt][2 * rr];
                    oo[(warp * GR + row) * D + nt * 8 + qcol + 1] = o[nt][2 * rr + 1];
                }
            }
        }
        named_bar_sync(1, 32 * C::kConsumers);
        for (int e = threadIdx.x; e < G * D; e += 32 * C::kConsumers) {
            const int row = e / D, d = e % D;
            float M = -INFINITY;
#pragma unroll
            for (int x = 0; x < C::kConsumers; ++x) M = fmaxf(M, mm[x * GR + row]);
            const float Mref = M == -INFINITY ? 0.f : M;
            float L = 0.f, acc = 0.f;
#pragma unroll
            for (int x = 0; x < C::kConsumers; ++x) {
                const float f = ex2_approx(mm[x * GR + row] - Mref);
                L += f * ll[x * GR + row];
                acc += f * oo[(x * GR + row) * D + d];
            }
            const int h = w.kvh * G + row;
            if (w.nsplit > 1) {
                const int64_t pr = (int64_t)w.pbase + (int64_t)h * w.nsplit + w.split;
                p.part_o[pr * D + d] = acc;
                if (d == 0)
                    reinterpret_cast<float2 *>(p.part_ml)[pr] = make_float2(M, L);
            } else {
                reinterpret_cast<__nv_bfloat16 *>(p.out)[((int64_t)w.t * p.num_q_heads + h) * D + d] =
                    __float2bfloat16_rn(L > 0.f ? acc / L : 0.f);
            }
        }
        named_bar_sync(1, 32 * C::kConsumers);
    }
    if (threadIdx.x == 0 && *abort)
        set_dev_error(p.dev_err, CPSA_DEV_WAIT_TIMEOUT);
}

template <int D, bool HI>
cudaError_t launch_decode_t(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv, int grid,
                            cudaStream_t s, bool early)
{
    using C = DecCfg<D, HI>;
    static std::atomic<uint64_t> done{0};
    auto k = decode_attn_kernel<D, HI>;
    return launch_with_smem(done, reinterpret_cast<const void *>(k), C::kSmemBytes, [&] {
        return launch_pdl(early, k, dim3(grid), dim3(C::kThreads), C::kSmemBytes, s, p, tk, tv);
    });
}


// ---------------------------------------------------------------------------
// Grouped decode: one item covers a group of HG kv heads (4 or 8) of one decode
// row, so its stages read every head of a page at once. The cache is
// [pages][Hkv][P][D]: the heads of a page are contiguous, and a whole-page read
// stream runs near the copy bandwidth (a copy-only probe of the Sarathi-sized
// cache: 6.9-7.1 TB/s), where one head's 4 KB block per page at a time does not
// (the per-head kernel above: about 5 TB/s even without its arithmetic).
// CTA: HG consumer warps, warp h owning kv head group * HG + h over all keys of
// the item (no merge between warps), then one producer warp.
// Stage: 16 keys of all HG heads, K and V, one TMA box per page (two at page 8)
// covering the heads and both 64-column halves of head_dim: a 5-D view of the
// cache (columns, rows, halves, heads, pages), 128-byte swizzled, landing as
// [box][head][half][rows][128 B]. One lane announces and issues all of a
// stage's copies. Page numbers of 32 stages are looked up at a time, the next
// window while the current one streams.
template <int D, int HG>
struct GDecCfg {
    static constexpr int kHalves = D / 64;
    static constexpr int kKeys = 16;                                  // keys per stage
    static constexpr int kTileBytes = HG * kKeys * D * 2;             // K (or V) of one stage
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kStagesRaw = 196608 / kStageBytes;
    static constexpr int kStages = kStagesRaw > 12 ? 12 : (kStagesRaw < 2 ? 2 : kStagesRaw);
    static constexpr int kBarOff = kStages * kStageBytes;
    static constexpr int kSmemBytes = kBarOff + 512 + 1024;
    static constexpr int kThreads = 32 * (HG + 1);
    static_assert(kSmemBytes <= 232448, "beyond the 227 KB of shared memory a CTA may have");
};

struct GDecBars {
    uint64_t full[12], empty[12];
    uint64_t patch;   // fused KV write: copies of the stage that gets the new row
    int abort;
};

// Byte address of element (key, head, col) of a grouped stage tile, boxes of
// 2^lgrb rows: [box][head][half][row][128 B], 16-byte chunks swizzled by the row.
template <int D, int HG>
__device__ __forceinline__ uint32_t gdec_addr(uint32_t base, int key, int head, int col, int lgrb)
{
    const int b = key >> lgrb, kr = key & ((1 << lgrb) - 1);
    const int c = col >> 6, ch = (col & 63) >> 3;
    return base + ((uint32_t)((b * HG + head) * (D / 64) + c) << (lgrb + 7)) + ((uint32_t)kr << 7) +
           ((ch ^ (kr & 7)) << 4) + (col & 7) * 2;
}

template <int D, int HG, bool HI>
__global__ void __launch_bounds__(GDecCfg<D, HG>::kThreads, 1)
decode_group_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v)
{
    using C = GDecCfg<D, HG>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    GDecBars *bars = reinterpret_cast<GDecBars *>(smem + C::kBarOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], HG);
        }
        mbar_init(&bars->patch, 1);
        bars->abort = 0;
        fence_barrier_init();
    }
    // set-up above touches no global memory: from here on the plan's output
    pdl_trigger();
    pdl_wait();
    const int n_items = p.counts[kCntDecode];
    __syncthreads();
    volatile int *abort = &bars->abort;
    const int RB = p.page_size < C::kKeys ? p.page_size : C::kKeys;   // rows per box: 8 or 16
    const int lgrb = RB == 8 ? 3 : 4;
    const int NBX = C::kKeys / RB;                                    // boxes per stage: 1 or 2

    if (warp == HG) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
        }
        const uint32_t box_bytes = (uint32_t)HG * RB * D * 2;
        uint32_t g = 0, patch_uses = 0;
        bool stop = false;
        // the next item's descriptor is read one item ahead (its page lookups
        // depend on it, and they start the item's stream)
        DecodeItem w_next{};
        if (blockIdx.x < n_items)
            w_next = p.ditems[blockIdx.x];
        for (int it = blockIdx.x; it < n_items && !stop && !*abort; it += gridDim.x) {
            const DecodeItem w = w_next;
            if (it + (int)gridDim.x < n_items)
                w_next = p.ditems[it + gridDim.x];
            const int32_t *bt_row = p.block_table + (int64_t)w.r * p.max_blocks;
            const int head0 = w.kvh * HG;
            // the row's own key, when this item's range ends with it and the KV write is fused
            const int knew = (p.fused && w.key1 == p.seq_lens[w.r]) ? w.key1 - 1 : -1;
            // lane j holds the page numbers of stage 32 m + j of window m (box 0, and box 1
            // at page 8); the next window's are loaded while the current one streams
            auto lookup = [&](int m, int b) -> int {
                const int key = w.key0 + (32 * m + lane) * C::kKeys + b * RB;
                return (b < NBX && key < w.key1) ? __ldg(bt_row + key / p.page_size) : -1;
            };
            int cur0 = lookup(0, 0), cur1 = lookup(0, 1);
            int nxt0 = lookup(1, 0), nxt1 = lookup(1, 1);
            int j = 0;
            for (int c0 = w.key0; c0 < w.key1; c0 += C::kKeys, ++g, ++j) {
                if (j > 0 && (j & 31) == 0) {
                    cur0 = nxt0;
                    cur1 = nxt1;
                    nxt0 = lookup((j >> 5) + 1, 0);
                    nxt1 = lookup((j >> 5) + 1, 1);
                }
                const int pg0 = __shfl_sync(0xffffffffu, cur0, j & 31);
                const int pg1 = __shfl_sync(0xffffffffu, cur1, j & 31);
                const int stage = g % C::kStages;
                if (g >= (uint32_t)C::kStages &&
                    !mbar_wait(&bars->empty[stage], ((g / C::kStages) - 1) & 1, abort)) {
                    stop = true;
                    break;
                }
                uint8_t *kdst = smem + stage * C::kStageBytes;
                uint8_t *vdst = kdst + C::kTileBytes;
                const bool patch = knew >= c0 && knew < c0 + C::kKeys;
                uint64_t *bar = patch ? &bars->patch : &bars->full[stage];
                if (lane == 0) {
                    // one lane announces the stage's bytes, then issues its copies
                    bool v0 = false, v1 = false;
                    if (c0 < w.key1) {
                        v0 = pg0 >= 0 && pg0 < p.num_pages;
                        if (!v0)
                            set_dev_error(p.dev_err, CPSA_DEV_PAGE_OUT_OF_RANGE);
                    }
                    if (NBX == 2 && c0 + RB < w.key1) {
                        v1 = pg1 >= 0 && pg1 < p.num_pages;
                        if (!v1)
                            set_dev_error(p.dev_err, CPSA_DEV_PAGE_OUT_OF_RANGE);
                    }
                    mbar_arrive_expect_tx(bar, (uint32_t)((v0 ? 2 : 0) + (v1 ? 2 : 0)) * box_bytes);
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        const bool vb = b == 0 ? v0 : v1;
                        if (!vb)
                            continue;
                        const int pg = b == 0 ? pg0 : pg1;
                        const int off = (c0 + b * RB) % p.page_size;
                        if (C::kHalves == 2) {
                            tma_load_5d(kdst + b * box_bytes, &tm_k, bar, 0, off, 0, head0, pg);
                            tma_load_5d(vdst + b * box_bytes, &tm_v, bar, 0, off, 0, head0, pg);
                        } else {
                            tma_load_4d(kdst + b * box_bytes, &tm_k, bar, 0, off, head0, pg);
                            tma_load_4d(vdst + b * box_bytes, &tm_v, bar, 0, off, head0, pg);
                        }
                    }
                }
                __syncwarp();
                if (patch) {
                    if (!mbar_wait(&bars->patch, patch_uses & 1u, abort)) {
                        stop = true;
                        break;
                    }
                    ++patch_uses;
                    // the new token's K and V rows of the HG heads, 16-byte chunks over the
                    // lanes: into the stage (over the cache's old bytes) and to the slot
                    const int rr = knew - c0;
                    const int64_t slot = __ldg(p.slot_mapping + w.t);
                    constexpr int CPR = D / 8;
                    for (int x = lane; x < 2 * HG * CPR; x += 32) {
                        const int which = x / (HG * CPR), rem = x - which * (HG * CPR);
                        const int h = rem / CPR, ch = rem - h * CPR;
                        const int64_t src = ((int64_t)w.t * p.num_kv_heads + head0 + h) * CPR + ch;
                        const uint4 val = __ldg(reinterpret_cast<const uint4 *>(which ? p.v_new : p.k_new) + src);
                        uint8_t *tile = which ? vdst : kdst;
                        *reinterpret_cast<uint4 *>(tile + (gdec_addr<D, HG>(0, rr, h, ch * 8, lgrb))) = val;
                        if (slot >= 0 && slot < p.num_pages * (int64_t)p.page_size) {
                            const int lg_p = __ffs(p.page_size) - 1;   // page_size is a power of two
                            const int64_t spg = slot >> lg_p, po = slot & (p.page_size - 1);
                            reinterpret_cast<uint4 *>(which ? p.v_cache_w : p.k_cache_w)
                                [((spg * p.num_kv_heads + head0 + h) * p.page_size + po) * CPR + ch] = val;
                        }
                    }
                    if (lane == 0 && slot >= p.num_pages * (int64_t)p.page_size)
                        set_dev_error(p.dev_err, CPSA_DEV_SLOT_OUT_OF_RANGE);
                    fence_proxy_async_smem();   // the patch before later copies into this stage
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&bars->full[stage]);
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // Warp h: kv head w.kvh * HG + h and its G q heads (the M rows of
    // mma.sync m16n8k16, rows >= G zero; rows lane/4 and, when HI, lane/4 + 8).
    constexpr int R = HI ? 2 : 1;
    const float sl2 = p.scale_log2;
    const int qrow = lane >> 2;
    const int qcol = (lane & 3) * 2;
    const int h = warp;
    uint32_t g = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const DecodeItem w = p.ditems[it];
        const int nch = (w.key1 - w.key0 + C::kKeys - 1) / C::kKeys;
        const int kvh = w.kvh * HG + h;
        uint32_t qa[D / 16][4];
        {
            const uint32_t *qsrc = reinterpret_cast<const uint32_t *>(
                reinterpret_cast<const __nv_bfloat16 *>(p.q) + ((int64_t)w.t * p.num_q_heads + kvh * G) * D);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int row = qrow + 8 * rr;
                    const bool live = (rr == 0 || HI) && row < G;
                    qa[kk][rr] = live ? __ldg(qsrc + (row * D + kk * 16 + qcol) / 2) : 0u;
                    qa[kk][2 + rr] = live ? __ldg(qsrc + (row * D + kk * 16 + 8 + qcol) / 2) : 0u;
                }
            }
        }
        float m_run[R], l_run[R];
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            m_run[rr] = -INFINITY;
            l_run[rr] = 0.f;
        }
        float o[D / 8][4];
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

        for (int j = 0; j < nch; ++j) {
            const uint32_t gg = g + j;
            const int stage = gg % C::kStages;
            if (!mbar_wait(&bars->full[stage], (gg / C::kStages) & 1, abort))
                break;
            const int c0 = w.key0 + j * C::kKeys;
            const int nv = min(C::kKeys, w.key1 - c0);   // valid keys of this stage (>= 1)
            uint8_t *kst = smem + stage * C::kStageBytes;
            uint8_t *vst = kst + C::kTileBytes;
            if (nv < C::kKeys) {
                // value rows past the range may hold anything (NaN included): zero this
                // head's (whole 128-byte half-rows, so the swizzle does not matter)
                const int nchunks = (C::kKeys - nv) * C::kHalves * 8;
                for (int x = lane; x < nchunks; x += 32) {
                    const int row = nv + x / (C::kHalves * 8);
                    const int half = (x >> 3) % C::kHalves;
                    const int b = row >> lgrb, kr = row & ((1 << lgrb) - 1);
                    *reinterpret_cast<uint4 *>(vst + (((b * HG + h) * C::kHalves + half) << (lgrb + 7)) + (kr << 7) +
                                               (x & 7) * 16) = make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            const uint32_t kb = smem_u32(kst), vb = smem_u32(vst);
            const int mat = lane >> 3, mrow = lane & 7;
            // S = q K^T over the stage's 16 keys: 2 n-tiles of 8
            float s[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(gdec_addr<D, HG>(kb, mrow + (mat >> 1) * 8, h, kk * 16 + (mat & 1) * 8, lgrb), b0, b1, b2, b3);
                mma_bf16(s[0], qa[kk], b0, b1);
                mma_bf16(s[1], qa[kk], b2, b3);
            }
            uint32_t pa[4];
            pa[0] = pa[1] = pa[2] = pa[3] = 0u;
#pragma unroll
            for (int rr = 0; rr < R; ++rr) {
                float mx = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        if (nt * 8 + qcol + e >= nv) s[nt][2 * rr + e] = -INFINITY;
                        mx = fmaxf(mx, s[nt][2 * rr + e]);
                    }
                }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float m_new = fmaxf(m_run[rr], mx * sl2);
                const float alpha = m_new == m_run[rr] ? 1.f : ex2_approx(m_run[rr] - m_new);
                m_run[rr] = m_new;
                const float mref = m_new == -INFINITY ? 0.f : m_new;
                float psum = 0.f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const float p0 = ex2_approx(fmaf(s[nt][2 * rr], sl2, -mref));
                    const float p1 = ex2_approx(fmaf(s[nt][2 * rr + 1], sl2, -mref));
                    psum += p0 + p1;
                    pa[nt * 2 + rr] = pack_bf16x2(p0, p1);
                }
                l_run[rr] = l_run[rr] * alpha + psum;
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt) {
                    o[nt][2 * rr] *= alpha;
                    o[nt][2 * rr + 1] *= alpha;
                }
            }
            // O += P V
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(gdec_addr<D, HG>(vb, mrow + (mat & 1) * 8, h, np * 16 + (mat >> 1) * 8, lgrb), b0, b1, b2,
                          b3);
                mma_bf16(o[2 * np], pa, b0, b1);
                mma_bf16(o[2 * np + 1], pa, b2, b3);
            }
            if (nv < C::kKeys)
                fence_proxy_async_smem();   // our zeroing writes before the next copy into this stage
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars->empty[stage]);
        }
        g += nch;
        // this warp's rows are complete: the bf16 row, or the split's partial
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            float lq = l_run[rr];
            lq += __shfl_xor_sync(0xffffffffu, lq, 1);
            lq += __shfl_xor_sync(0xffffffffu, lq, 2);
            const int row = qrow + 8 * rr;
            if (row >= G)
                continue;
            const int hq = kvh * G + row;
            if (w.nsplit > 1) {
                const int64_t pr = (int64_t)w.pbase + (int64_t)hq * w.nsplit + w.split;
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt)
                    *reinterpret_cast<float2 *>(p.part_o + pr * D + nt * 8 + qcol) =
                        make_float2(o[nt][2 * rr], o[nt][2 * rr + 1]);
                if ((lane & 3) == 0)
                    reinterpret_cast<float2 *>(p.part_ml)[pr] = make_float2(m_run[rr], lq);
            } else {
                const float inv = lq > 0.f ? 1.f / lq : 0.f;
                uint32_t *dst = reinterpret_cast<uint32_t *>(reinterpret_cast<__nv_bfloat16 *>(p.out) +
                                                             ((int64_t)w.t * p.num_q_heads + hq) * D + qcol);
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt)
                    dst[nt * 4] = pack_bf16x2(o[nt][2 * rr] * inv, o[nt][2 * rr + 1] * inv);
            }
        }
    }
    if (threadIdx.x == 0 && *abort)
        set_dev_error(p.dev_err, CPSA_DEV_WAIT_TIMEOUT);
}

template <int D, int HG, bool HI>
cudaError_t launch_decode_group_t(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv, int grid,
                                  cudaStream_t s, bool early)
{
    using C = GDecCfg<D, HG>;
    static std::atomic<uint64_t> done{0};
    auto k = decode_group_kernel<D, HG, HI>;
    return launch_with_smem(done, reinterpret_cast<const void *>(k), C::kSmemBytes, [&] {
        return launch_pdl(early, k, dim3(grid), dim3(C::kThreads), C::kSmemBytes, s, p, tk, tv);
    });
}

template <int HG>
cudaError_t launch_decode_group_hg(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv, int head_dim,
                                   int grid, cudaStream_t s, bool early)
{
    if (p.group > 8)
        return head_dim == 128 ? launch_decode_group_t<128, HG, true>(p, tk, tv, grid, s, early)
                               : launch_decode_group_t<64, HG, true>(p, tk, tv, grid, s, early);
    return head_dim == 128 ? launch_decode_group_t<128, HG, false>(p, tk, tv, grid, s, early)
                           : launch_decode_group_t<64, HG, false>(p, tk, tv, grid, s, early);
}

}  // namespace

cudaError_t launch_decode_attn(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv, int head_dim,
                               int grid, cudaStream_t s, bool early)
{
    if (p.group > 8)
        return head_dim == 128 ? launch_decode_t<128, true>(p, tk, tv, grid, s, early)
                               : launch_decode_t<64, true>(p, tk, tv, grid, s, early);
    return head_dim == 128 ? launch_decode_t<128, false>(p, tk, tv, grid, s, early)
                           : launch_decode_t<64, false>(p, tk, tv, grid, s, early);
}

cudaError_t launch_decode_group(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv, int head_dim,
                                int heads_per_item, int grid, cudaStream_t s, bool early)
{
    return heads_per_item == 8 ? launch_decode_group_hg<8>(p, tk, tv, head_dim, grid, s, early)
                               : launch_decode_group_hg<4>(p, tk, tv, head_dim, grid, s, early);
}

}  // namespace cpsa
