// plan.cuh -- work items and workspace layout shared by the metadata kernel and
// the attention kernels.
//
// One call of cpp_chunked_prefill_attn runs:
//   plan      one CTA (one warp for up to 32 requests): scan of query_lens,
//             validation, work lists, split choice
//   chunk     tensor-core kernel over prefill items (query_len >= 2); merges
//             the units the stream-K cut split
//   decode    split-KV kernel over decode items (query_len == 1)
//   combine   merges the partial results of decode rows split along keys
// The lists live in the caller's workspace; every kernel is persistent and reads
// its item count from the workspace, so the host never needs the lengths. A
// batch of one prefill request of at most about 6.6k tokens (32/8 heads, 152
// SMs) runs the chunk kernel alone: its CTAs compute their own runs (same units
// and cuts as the plan).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace cpsa {

// Split policy.
// Prefill: stream-K. The KV tiles of all prefill units (one unit = a 128-row
// query tile x kv head x head pair) are laid end to end and cut into equal runs
// of max(ceil(W / grid), kMinRunTiles) tiles, one run per CTA of the chunk
// kernel; a unit cut by a run boundary becomes several pieces, merged inside the
// chunk kernel by whichever piece finishes last (a counter per unit and q head;
// no CTA waits for another). Every CTA gets the same amount of work, counting
// for every unit kUnitCostTiles positions ahead of its tiles: the fixed cost of
// starting and finishing an item (loading its Q, storing its rows), which a run
// of many short units pays many times. Those positions hold no tile: a unit's
// first piece belongs to the run that holds its first tile.
// Decode: a row splits into pieces of kDecodeKeysPerSplit keys (grouped items:
// kDecodeKeysPerSplitGrouped) (at most
// max_kv_splits), depending only on its own length.
// KV tiles of a unit: tile kt holds keys [128 kt, 128 kt + 128). With the KV
// write fused, the history (keys below h) keeps that grid, its last tile cut at
// h, and the chunk's own keys form tiles of their own starting at h, so that
// they come from the new K/V rows: tile ceil(h / 128) + j holds keys
// [h + 128 j, h + 128 j + 128), and the unit of query tile i has ceil(h / 128) +
// i + 1 tiles (the same count whenever h is a multiple of 128).
constexpr int kMinRunTiles = 4;             // shortest run of KV tiles per CTA
#ifndef CPSA_UNIT_COST_TILES
#define CPSA_UNIT_COST_TILES 2
#endif
constexpr int kUnitCostTiles = CPSA_UNIT_COST_TILES;   // a unit's fixed cost, in KV tiles (< kMinRunTiles)
static_assert(kUnitCostTiles >= 0 && kUnitCostTiles < kMinRunTiles, "a run must hold more than one unit's start");
constexpr int kCutCostTiles = 6;            // a run's extra item and merge when a unit is cut, in KV tiles
constexpr int kMaxChunkGrid = 256;          // upper bound of the chunk kernel's grid (SMs)
constexpr int kDecodeChunk = 64;            // keys per decode pipeline stage
constexpr int kDecodeKeysPerSplit = 4096;   // keys per decode split (multiple of kDecodeChunk)
// Grouped decode items carry all heads of a group, a quarter to an eighth of the
// per-head items' count: they split every 1024 keys so that small decode batches
// still occupy the GPU (still a function of the row's own length only).
constexpr int kDecodeKeysPerSplitGrouped = 1024;
constexpr int kMaxSplitUnits = kMaxChunkGrid;   // a split unit holds a run boundary: at most grid - 1
constexpr int kMergeCounters = 2 * 4;          // per split unit: q heads (<= 2) x 4 softmax warps
// A batch of one prefill request skips the plan kernel: every chunk-kernel CTA
// computes its own run's pieces (at most this many, kept in shared memory).
constexpr int kSelfPlanCap = 56;

// A prefill piece: KV tiles [kt0, kt1) of the unit (request r, query tile at
// row i0, kv head kvh, head pair hp); piece `piece` of `npieces` of that unit.
// aux: for a whole unit (npieces = 1) the CTA that processes it; for a piece of
// a split unit, the unit's ordinal among the batch's split units (its merge
// counters), its partial rows at pbase.
struct alignas(16) PrefillItem {
    int32_t r, i0, kvh_hp, kt0, kt1, piece_np, pbase, aux;
};

// A decode item: the single new token (global row t) of request r, all q heads
// of kv head kvh (the grouped decode kernel: of kv heads kvh * dec_heads ..
// kvh * dec_heads + dec_heads - 1), keys [key0, key1) of split `split`.
struct DecodeItem {
    int32_t r, kvh, key0, key1, split, nsplit, pbase, t;
};

// Split decode rows for the combine kernel.
// Rows [t0, t0 + nrows) x q heads [h0, h0 + nh) had nsplit partials each:
// unit u = row * nh + (head - h0) at pbase + u * nsplit + s.
// u0: number of (row, head) units of all earlier combine items.
struct CombineItem {
    int32_t t0, nrows, h0, nh, pbase, nsplit, u0, pad;
};

enum CountSlot {
    kCntPrefill = 0,
    kCntDecode = 1,
    kCntCombine = 2,
    kCntPartialRows = 3,
    kCntCombineUnits = 4,
    kCntRunTiles = 5,
    kCntSplitUnits = 6,
    kCntSlots = 16
};

struct WsLayout {
    size_t off_counts, off_cuq, off_runs, off_flags, off_pitems, off_ditems, off_citems, off_pml, off_po, end_meta,
        end_full;
    int64_t max_pitems, max_ditems, max_citems, max_prows_full;
};

__host__ __device__ inline size_t ws_align(size_t x) { return (x + 255) & ~(size_t)255; }

// Upper bounds of the work lists for a batch of num_reqs requests and num_tokens
// new tokens (every prefill request has >= 2 tokens, so at most num_tokens/2).
inline WsLayout ws_layout(int num_reqs, int64_t num_tokens, int Hq, int Hkv, int D, int max_splits,
                          int nq_per_cta)
{
    WsLayout L{};
    int64_t B = num_reqs, T = num_tokens;
    int64_t nprefill = B < T / 2 ? B : T / 2;
    int64_t ndecode = B < T ? B : T;
    int64_t qtiles = T / 128 + nprefill + 1;
    int64_t units = qtiles * Hkv * ((Hq / Hkv) / nq_per_cta);
    L.max_pitems = units + kMaxChunkGrid;
    L.max_ditems = ndecode * Hkv * max_splits;
    L.max_citems = ndecode;   // split decode rows
    // prefill: a cut inside a unit adds one piece, at most 2 pieces' partials per cut
    const int64_t prefill_rows = max_splits > 1 ? (int64_t)2 * kMaxChunkGrid * 128 * nq_per_cta : 0;
    const int64_t decode_rows = max_splits > 1 ? ndecode * Hq * max_splits : 0;
    L.max_prows_full = prefill_rows + decode_rows;
    size_t o = 0;
    L.off_counts = o; o = ws_align(o + sizeof(int32_t) * kCntSlots);
    L.off_cuq = o;    o = ws_align(o + sizeof(int32_t) * (size_t)(B + 1));
    L.off_runs = o;   o = ws_align(o + sizeof(int32_t) * (size_t)(kMaxChunkGrid + 1));
    L.off_flags = o;  o = ws_align(o + sizeof(unsigned long long) * (size_t)kMaxSplitUnits * kMergeCounters);
    L.off_pitems = o; o = ws_align(o + sizeof(PrefillItem) * (size_t)L.max_pitems);
    L.off_ditems = o; o = ws_align(o + sizeof(DecodeItem) * (size_t)L.max_ditems);
    L.off_citems = o; o = ws_align(o + sizeof(CombineItem) * (size_t)L.max_citems);
    L.end_meta = o;
    L.off_pml = o;
    size_t ml = ws_align(sizeof(float) * 2 * (size_t)L.max_prows_full);
    L.off_po = o + ml;
    L.end_full = L.off_po + ws_align(sizeof(float) * (size_t)D * (size_t)L.max_prows_full);
    return L;
}

// Partial-row capacity that fits in `bytes` of workspace (m,l pairs + D floats each).
inline int64_t ws_partial_capacity(const WsLayout &L, size_t bytes, int D)
{
    if (bytes <= L.end_meta + 512)
        return 0;
    size_t room = bytes - L.end_meta - 512;
    return (int64_t)(room / (sizeof(float) * (2 + (size_t)D)));
}

struct PlanParams {
    const int32_t *query_lens;
    const int32_t *seq_lens;
    int num_reqs;
    int64_t num_tokens;
    int max_blocks;
    int page_size;
    int Hq, Hkv, group, nq;    // nq: q heads per chunk-kernel CTA (1 or 2)
    int max_splits;
    int dec_heads;             // kv heads per decode item: 1, or a group of 4 or 8 (the grouped decode kernel)
    int chunk_grid;            // CTAs of the chunk kernel (stream-K runs)
    int fused;                 // KV write fused: the chunk's own keys form tiles of their own
    int64_t prow_capacity;     // partial rows that fit
    int32_t *counts;
    int32_t *cu_q;
    int32_t *run_first;        // [chunk_grid + 1]: first piece of each CTA's run
    unsigned long long *flags; // [kMaxSplitUnits][nq][4]: merge counters (epoch-tagged, see ChunkParams)
    PrefillItem *pitems;
    DecodeItem *ditems;
    CombineItem *citems;
    int64_t max_pitems, max_ditems, max_citems;
    uint32_t *dev_err;
};

cudaError_t launch_plan(const PlanParams &p, cudaStream_t s, bool early = true);

}  // namespace cpsa
