// kernels.cuh -- parameter blocks and launchers of the attention-step kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "plan.cuh"

namespace cpsa {

// Fields common to the chunk (prefill) and decode kernels.
struct AttnCommon {
    const int32_t *counts;
    const int32_t *cu_q;
    const int32_t *query_lens;
    const int32_t *seq_lens;
    const int32_t *block_table;
    int max_blocks;
    int page_size;
    int64_t num_pages;
    int num_q_heads, num_kv_heads, group;
    float scale_log2;          // scale * log2(e): scores go straight to the base-2 exponent
    void *out;                 // bf16 [T][Hq][D]
    float *part_o;             // [rows][D] fp32 partial outputs of split rows (prefill pieces: O / l in bf16 in the same pitch)
    float *part_ml;            // fp32 [rows][2]  (max in log2 units, row sum)
    uint32_t *dev_err;
    // KV write fused into the attention (fused != 0): the new tokens' keys and
    // values are read from k_new / v_new rather than from the cache, and each is
    // also stored, once, to the cache slot slot_mapping names
    int fused;
    const void *k_new, *v_new;         // bf16 [T][Hkv][D]
    const int64_t *slot_mapping;       // [T]
    void *k_cache_w, *v_cache_w;       // bf16 [pages][Hkv][P][D], written
};

struct ChunkParams : AttnCommon {
    const PrefillItem *pitems;
    const int32_t *run_first;   // CTA c processes pieces [run_first[c], run_first[c + 1])
    // Merge counters, per split unit, q head and softmax warp: the pieces of the
    // unit done in this call, tagged with the call's epoch in the high 32 bits.
    // The warp that merges a unit clears its counter; a count that an earlier
    // call left (it ended early) carries another epoch and reads as zero, so
    // nothing has to clear the counters between calls.
    unsigned long long *flags;
    uint32_t epoch;             // nonzero, different for every call of the library
    // A batch of one prefill request (self_plan != 0): no plan kernel ran; every
    // CTA computes its own run's pieces from query_lens[0] / seq_lens[0].
    int self_plan;
    int num_tokens;             // for the self-planned batch's token check
    int split_ok;               // self-planned batch: units may be cut (splits allowed and the partials fit)
    int split_clamped;          // self-planned batch: splits were asked for but the partials do not fit
    int out_tma;                // head_dim 128, `out` mapped for TMA stores (whole units' rows without the KV
                                // write, merged rows at the end of a run)
};

struct DecodeParams : AttnCommon {
    const DecodeItem *ditems;
    const void *q;             // bf16 [T][Hq][D]
    const void *k_cache_ptr;   // bf16 [pages][Hkv][P][D]
    const void *v_cache_ptr;
};

struct CombineParams {
    const int32_t *counts;
    const CombineItem *citems;
    const float *part_o;
    const float *part_ml;
    void *out;
    int num_q_heads;
};

// early: launch with programmatic dependent launch (see launch_pdl)
// tkn / tvn: maps over k_new / v_new (used when p.fused)
// to: map over out, boxes of 64 columns x 1 head x 32 rows (used when p.out_tma)
// tv4: 4-D map over v_cache, one box per page with both column halves (used for
//      head_dim 128 below page 128)
cudaError_t launch_chunk_attn(const ChunkParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                              const CUtensorMap &tv, const CUtensorMap &tkn, const CUtensorMap &tvn,
                              const CUtensorMap &to, const CUtensorMap &tv4, int head_dim, int nq, int grid,
                              cudaStream_t s, bool early);
cudaError_t launch_decode_attn(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv, int head_dim,
                               int grid, cudaStream_t s, bool early);
// the grouped decode kernel: items of heads_per_item (4 or 8) kv heads; tk / tv
// are the grouped views of the caches (see abi.cu: make_map_group)
cudaError_t launch_decode_group(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv, int head_dim,
                                int heads_per_item, int grid, cudaStream_t s, bool early);
cudaError_t launch_combine(const CombineParams &p, int head_dim, int grid, cudaStream_t s, bool early);

cudaError_t launch_kv_cache_write(const void *k, const void *v, const int64_t *slot_mapping,
                                  int64_t num_tokens, int num_kv_heads, int head_dim,
                                  int page_size, int64_t num_pages, void *k_cache, void *v_cache,
                                  uint32_t *dev_err, int num_sms, cudaStream_t s);
cudaError_t launch_split_microbatch(const int32_t *query_lens, int num_reqs, float balance_threshold,
                                    int32_t length_threshold, int32_t *out3, cudaStream_t s);

cudaError_t launch_exp2_selftest(const float *x, float *poly, float *hw, int64_t n, cudaStream_t s);
cudaError_t launch_wait_selftest(uint64_t limit_ns, uint32_t *dev_err, int32_t *out, cudaStream_t s);


}  // namespace cpsa
