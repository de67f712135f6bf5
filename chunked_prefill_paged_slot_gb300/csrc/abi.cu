// abi.cu -- the extern "C" entry points of libcpsa.so (declared in
// include/cpsa.h): argument checks, TMA tensor maps, workspace carving and the
// stream-ordered launch sequence. No device memory is allocated here.
#include <math.h>
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.cuh"
#include "plan.cuh"

using namespace cpsa;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

// SM count of the current device (cached per device ordinal).
int sm_count()
{
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0)
        return 0;
    if (dev < 64 && cache[dev])
        return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    if (dev < 64)
        cache[dev] = n;
    return n;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool pow2_in(int x, int lo, int hi) { return x >= lo && x <= hi && (x & (x - 1)) == 0; }

// 3-D bf16 tensor map, innermost dimension first, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1_bytes,
              uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2)
{
    auto enc = encode_fn();
    if (!enc)
        return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 4-D bf16 view of a head_dim-128 cache, [cols 64][rows page][half 2][page-head
// blocks], halves 128 bytes apart: one box of `rows` rows x both halves lands as
// [half][rows][128 B] with the 128-byte swizzle.
bool make_map4_halves(CUtensorMap *m, const void *base, int page_size, uint64_t blocks, uint32_t rows)
{
    auto enc = encode_fn();
    if (!enc)
        return false;
    cuuint64_t dims[4] = {64, (cuuint64_t)page_size, 2, blocks};
    cuuint64_t strides[3] = {256, 128, (cuuint64_t)page_size * 256};
    cuuint32_t box[4] = {64, rows, 2, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// View of a cache [pages][Hkv][P][D] for the grouped decode kernel, innermost
// dimension first: 64 columns, P rows, (2 halves of head_dim 128,) Hkv heads,
// pages. A box of `rows` rows of `heads` consecutive heads (both halves) lands as
// [head][half][rows][128 B], 128-byte swizzled.
bool make_map_group(CUtensorMap *m, const void *base, int head_dim, int page_size, int num_kv_heads,
                    int64_t num_pages, uint32_t rows, uint32_t heads)
{
    auto enc = encode_fn();
    if (!enc)
        return false;
    const uint64_t row_bytes = (uint64_t)head_dim * 2;
    const uint64_t head_bytes = row_bytes * (uint64_t)page_size;
    CUresult r;
    if (head_dim == 128) {
        cuuint64_t dims[5] = {64, (cuuint64_t)page_size, 2, (cuuint64_t)num_kv_heads, (cuuint64_t)num_pages};
        cuuint64_t strides[4] = {row_bytes, 128, head_bytes, head_bytes * (uint64_t)num_kv_heads};
        cuuint32_t box[5] = {64, rows, 2, heads, 1};
        cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cuuint64_t dims[4] = {64, (cuuint64_t)page_size, (cuuint64_t)num_kv_heads, (cuuint64_t)num_pages};
        cuuint64_t strides[3] = {row_bytes, head_bytes, head_bytes * (uint64_t)num_kv_heads};
        cuuint32_t box[4] = {64, rows, heads, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS;
}

// kv heads per decode item: groups of 8 (else 4) heads read every page's heads
// together (the grouped decode kernel); 1 for other head counts.
int decode_heads_per_item(int num_kv_heads)
{
    return num_kv_heads % 8 == 0 ? 8 : (num_kv_heads % 4 == 0 ? 4 : 1);
}

int nq_for_group(int group) { return (group % 2 == 0) ? 2 : 1; }

// Every attention call gets its own nonzero epoch: the merge counters it leaves
// in the workspace carry it, so the next call tells them apart from its own.
std::atomic<uint32_t> g_epoch{0};

uint32_t next_epoch()
{
    uint32_t e;
    do {
        e = g_epoch.fetch_add(1u, std::memory_order_relaxed) + 1u;
    } while (e == 0u);
    return e;
}

// Whether a batch of one prefill request of num_tokens tokens can skip the plan
// kernel: every chunk-kernel run must fit its pieces in kSelfPlanCap. A run of R
// tiles holds at most (R - 2) / L + 2 pieces, L the shortest unit; that ratio is
// largest with no history (L = 1, R = R0, every unit as short as it gets) and
// stays below R0 + 3 for any history (the units grow as fast as the run).
bool self_plan_fits(int64_t num_tokens, int units_per_qtile, int grid)
{
    // the most pieces a run can hold is in the no-history case (the shortest
    // units): a run of r0 positions meets at most r0 / (1 + kUnitCostTiles) + 2 units
    // (each unit takes at least one tile and its fixed cost, plus the ones it starts
    // and ends inside); one more for safety
    const int64_t nqt = (num_tokens + kTileM - 1) / kTileM;
    const int64_t w0 = (int64_t)units_per_qtile * (nqt * (nqt + 1) / 2 + nqt * kUnitCostTiles);
    int64_t r0 = (w0 + grid - 1) / grid;
    if (r0 < kMinRunTiles)
        r0 = kMinRunTiles;
    return r0 / (1 + kUnitCostTiles) + 3 <= kSelfPlanCap;
}

int attn_impl(const void *q, const void *k_new, const void *v_new, const int64_t *slot_mapping, void *k_cache,
              void *v_cache, const int32_t *query_lens, const int32_t *seq_lens, const int32_t *block_table,
              int num_reqs, int64_t num_tokens, int max_blocks_per_req, int num_q_heads, int num_kv_heads,
              int head_dim, int page_size, int64_t num_pages, float scale, int max_kv_splits, void *out,
              void *workspace, size_t workspace_bytes, uint32_t *dev_err, void *stream, void *const *events);

int check_attn_shape(int num_reqs, int64_t num_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                     int max_kv_splits)
{
    if (num_reqs < 0 || num_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_kv_splits < 1 ||
        max_kv_splits > 32 || num_tokens > (int64_t)INT32_MAX / 2 || num_reqs >= (1 << 24))
        return CPSA_ERR_BAD_SHAPE;
    if (head_dim != 64 && head_dim != 128)
        return CPSA_ERR_UNSUPPORTED;
    if (num_q_heads % num_kv_heads != 0 || num_q_heads / num_kv_heads > kMaxGroup || num_q_heads > 65535)
        return CPSA_ERR_UNSUPPORTED;
    return CPSA_OK;
}

}  // namespace

extern "C" {

const char *cpp_status_string(int status)
{
    switch (status) {
    case CPSA_OK: return "ok";
    case CPSA_ERR_NULL_ARG: return "null argument";
    case CPSA_ERR_BAD_SHAPE: return "bad shape or count";
    case CPSA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case CPSA_ERR_UNSUPPORTED: return "unsupported head_dim, head grouping or page_size";
    case CPSA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case CPSA_ERR_CUDA: return "CUDA error";
    case CPSA_ERR_NO_DEVICE: return "no usable device";
    case CPSA_ERR_SCRATCH_TOO_SMALL: return "batch needs more than the library's built-in scratch area";
    case CPSA_ERR_SCRATCH_UNAVAILABLE:
        return "the library's built-in scratch area could not be reserved (device memory exhausted when its "
               "device code was loaded?)";
    default: return "unknown status";
    }
}

int cpp_kv_cache_write(const void *k, const void *v, const int64_t *slot_mapping, int64_t num_tokens,
                       int num_kv_heads, int head_dim, int page_size, int64_t num_pages, void *k_cache,
                       void *v_cache, uint32_t *dev_err, void *stream)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || num_pages < 0)
        return CPSA_ERR_BAD_SHAPE;
    if (head_dim != 64 && head_dim != 128)
        return CPSA_ERR_UNSUPPORTED;
    if (!pow2_in(page_size, 1, 1 << 20))
        return CPSA_ERR_UNSUPPORTED;
    if (num_tokens == 0)
        return CPSA_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache || !dev_err)
        return CPSA_ERR_NULL_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
        return CPSA_ERR_MISALIGNED;
    int sms = sm_count();
    if (sms <= 0)
        return CPSA_ERR_NO_DEVICE;
    cudaError_t e = launch_kv_cache_write(k, v, slot_mapping, num_tokens, num_kv_heads, head_dim, page_size,
                                          num_pages, k_cache, v_cache, dev_err, sms, (cudaStream_t)stream);
    return e == cudaSuccess ? CPSA_OK : CPSA_ERR_CUDA;
}

size_t cpp_attn_workspace_bytes(int num_reqs, int64_t num_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                                int max_kv_splits)
{
    if (check_attn_shape(num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim, max_kv_splits) != CPSA_OK)
        return 0;
    WsLayout L = ws_layout(num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim, max_kv_splits,
                           nq_for_group(num_q_heads / num_kv_heads));
    return L.end_full + 512;
}

size_t cpp_attn_workspace_min_bytes(int num_reqs, int64_t num_tokens, int num_q_heads, int num_kv_heads,
                                    int head_dim, int max_kv_splits)
{
    if (check_attn_shape(num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim, max_kv_splits) != CPSA_OK)
        return 0;
    WsLayout L = ws_layout(num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim, max_kv_splits,
                           nq_for_group(num_q_heads / num_kv_heads));
    return L.end_meta;
}

int cpp_chunked_prefill_attn(const void *q, const void *k_cache, const void *v_cache, const int32_t *query_lens,
                             const int32_t *seq_lens, const int32_t *block_table, int num_reqs, int64_t num_tokens,
                             int max_blocks_per_req, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                             int64_t num_pages, float scale, int max_kv_splits, void *out, void *workspace,
                             size_t workspace_bytes, uint32_t *dev_err, void *stream)
{
    return cpp_chunked_prefill_attn_events(q, k_cache, v_cache, query_lens, seq_lens, block_table, num_reqs,
                                           num_tokens, max_blocks_per_req, num_q_heads, num_kv_heads, head_dim,
                                           page_size, num_pages, scale, max_kv_splits, out, workspace,
                                           workspace_bytes, dev_err, stream, nullptr);
}

int cpp_chunked_prefill_attn_events(const void *q, const void *k_cache, const void *v_cache,
                                    const int32_t *query_lens, const int32_t *seq_lens, const int32_t *block_table,
                                    int num_reqs, int64_t num_tokens, int max_blocks_per_req, int num_q_heads,
                                    int num_kv_heads, int head_dim, int page_size, int64_t num_pages, float scale,
                                    int max_kv_splits, void *out, void *workspace, size_t workspace_bytes,
                                    uint32_t *dev_err, void *stream, void *const *events)
{
    return attn_impl(q, nullptr, nullptr, nullptr, const_cast<void *>(k_cache), const_cast<void *>(v_cache),
                     query_lens, seq_lens, block_table, num_reqs, num_tokens, max_blocks_per_req, num_q_heads,
                     num_kv_heads, head_dim, page_size, num_pages, scale, max_kv_splits, out, workspace,
                     workspace_bytes, dev_err, stream, events);
}

int cpp_chunked_prefill_attn_write_kv(const void *q, const void *k, const void *v, const int64_t *slot_mapping,
                                      void *k_cache, void *v_cache, const int32_t *query_lens,
                                      const int32_t *seq_lens, const int32_t *block_table, int num_reqs,
                                      int64_t num_tokens, int max_blocks_per_req, int num_q_heads, int num_kv_heads,
                                      int head_dim, int page_size, int64_t num_pages, float scale, int max_kv_splits,
                                      void *out, void *workspace, size_t workspace_bytes, uint32_t *dev_err,
                                      void *stream)
{
    return cpp_chunked_prefill_attn_write_kv_events(q, k, v, slot_mapping, k_cache, v_cache, query_lens, seq_lens,
                                                    block_table, num_reqs, num_tokens, max_blocks_per_req,
                                                    num_q_heads, num_kv_heads, head_dim, page_size, num_pages, scale,
                                                    max_kv_splits, out, workspace, workspace_bytes, dev_err, stream,
                                                    nullptr);
}

int cpp_chunked_prefill_attn_write_kv_events(const void *q, const void *k, const void *v,
                                             const int64_t *slot_mapping, void *k_cache, void *v_cache,
                                             const int32_t *query_lens, const int32_t *seq_lens,
                                             const int32_t *block_table, int num_reqs, int64_t num_tokens,
                                             int max_blocks_per_req, int num_q_heads, int num_kv_heads,
                                             int head_dim, int page_size, int64_t num_pages, float scale,
                                             int max_kv_splits, void *out, void *workspace,
                                             size_t workspace_bytes, uint32_t *dev_err, void *stream,
                                             void *const *events)
{
    if (num_tokens > 0 && (!k || !v || !slot_mapping))
        return CPSA_ERR_NULL_ARG;
    if ((k && !aligned16(k)) || (v && !aligned16(v)))
        return CPSA_ERR_MISALIGNED;
    return attn_impl(q, k, v, slot_mapping, k_cache, v_cache, query_lens, seq_lens, block_table, num_reqs,
                     num_tokens, max_blocks_per_req, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                     scale, max_kv_splits, out, workspace, workspace_bytes, dev_err, stream, events);
}

}  // extern "C"

namespace {

// The attention call; k_new != nullptr fuses the KV write (k_new, v_new,
// slot_mapping non-null then).
int attn_impl(const void *q, const void *k_new, const void *v_new, const int64_t *slot_mapping, void *k_cache,
              void *v_cache, const int32_t *query_lens, const int32_t *seq_lens, const int32_t *block_table,
              int num_reqs, int64_t num_tokens, int max_blocks_per_req, int num_q_heads, int num_kv_heads,
              int head_dim, int page_size, int64_t num_pages, float scale, int max_kv_splits, void *out,
              void *workspace, size_t workspace_bytes, uint32_t *dev_err, void *stream, void *const *events)
{
    const bool fused = k_new != nullptr;
    cudaEvent_t ev[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
    if (events)
        for (int i = 0; i < 5; ++i)
            ev[i] = static_cast<cudaEvent_t>(events[i]);
    // under stream capture a mark becomes an event node of the graph (recorded at
    // every replay); the external flag is for capture only
    auto mark = [&](int i, cudaStream_t st) {
        if (!ev[i])
            return;
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
            cudaEventRecordWithFlags(ev[i], st, cudaEventRecordExternal);
        else
            cudaEventRecord(ev[i], st);
    };
    // programmatic dependent launch between the call's own kernels, except when
    // events are recorded between them (each kernel then runs in plain stream
    // order); the call's first kernel always launches in plain stream order
    const bool early = events == nullptr;
    int st = check_attn_shape(num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim, max_kv_splits);
    if (st != CPSA_OK)
        return st;
    if (!pow2_in(page_size, 8, 256))
        return CPSA_ERR_UNSUPPORTED;
    if (max_blocks_per_req < 0 || num_pages < 0 || num_pages * num_kv_heads >= (int64_t)1 << 31)
        return CPSA_ERR_BAD_SHAPE;
    if (num_reqs == 0 || num_tokens == 0)
        return num_tokens == 0 ? CPSA_OK : CPSA_ERR_BAD_SHAPE;
    if (!q || !k_cache || !v_cache || !query_lens || !seq_lens || !block_table || !out || !workspace || !dev_err)
        return CPSA_ERR_NULL_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(workspace))
        return CPSA_ERR_MISALIGNED;
    const int group = num_q_heads / num_kv_heads;
    const int nq = nq_for_group(group);
    WsLayout L = ws_layout(num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim, max_kv_splits, nq);
    if (workspace_bytes < L.end_meta)
        return CPSA_ERR_WORKSPACE_TOO_SMALL;
    int64_t cap = max_kv_splits > 1 ? ws_partial_capacity(L, workspace_bytes, head_dim) : 0;
    if (cap > L.max_prows_full)
        cap = L.max_prows_full;
    const int sms = sm_count();
    if (sms <= 0)
        return CPSA_ERR_NO_DEVICE;
    if (num_pages == 0)
        return CPSA_ERR_BAD_SHAPE;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *counts = reinterpret_cast<int32_t *>(ws + L.off_counts);
    int32_t *cu_q = reinterpret_cast<int32_t *>(ws + L.off_cuq);
    int32_t *run_first = reinterpret_cast<int32_t *>(ws + L.off_runs);
    unsigned long long *flags = reinterpret_cast<unsigned long long *>(ws + L.off_flags);
    PrefillItem *pitems = reinterpret_cast<PrefillItem *>(ws + L.off_pitems);
    DecodeItem *ditems = reinterpret_cast<DecodeItem *>(ws + L.off_ditems);
    CombineItem *citems = reinterpret_cast<CombineItem *>(ws + L.off_citems);
    float *part_ml = reinterpret_cast<float *>(ws + L.end_meta);
    float *part_o = reinterpret_cast<float *>(ws + L.end_meta + ws_align(sizeof(float) * 2 * (size_t)cap));
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    PlanParams pp{};
    pp.query_lens = query_lens;
    pp.seq_lens = seq_lens;
    pp.num_reqs = num_reqs;
    pp.num_tokens = num_tokens;
    pp.max_blocks = max_blocks_per_req;
    pp.page_size = page_size;
    pp.Hq = num_q_heads;
    pp.Hkv = num_kv_heads;
    pp.group = group;
    pp.nq = nq;
    pp.max_splits = max_kv_splits;
    const int dec_heads = decode_heads_per_item(num_kv_heads);
    pp.dec_heads = dec_heads;
    pp.chunk_grid = sms < kMaxChunkGrid ? sms : kMaxChunkGrid;
    pp.fused = fused ? 1 : 0;
    pp.prow_capacity = cap;
    pp.counts = counts;
    pp.cu_q = cu_q;
    pp.run_first = run_first;
    pp.flags = flags;
    pp.pitems = pitems;
    pp.ditems = ditems;
    pp.citems = citems;
    pp.max_pitems = L.max_pitems;
    pp.max_ditems = L.max_ditems;
    pp.max_citems = L.max_citems;
    pp.dev_err = dev_err;
    // A single request is either one decode row or one prefill: the other
    // kernel would find no items, so it is not launched. A single prefill that
    // fits self-planning needs no plan kernel either: the chunk kernel's CTAs
    // compute their runs themselves, and it is the call's first kernel.
    const bool single_prefill = num_reqs == 1 && num_tokens >= 2;
    const bool single_decode = num_reqs == 1 && num_tokens == 1;
    const bool self_plan = single_prefill && self_plan_fits(num_tokens, num_kv_heads * (group / nq), pp.chunk_grid);
    mark(0, s);
    if (!self_plan && launch_plan(pp, s, false) != cudaSuccess)
        return CPSA_ERR_CUDA;
    mark(1, s);

    const float sc = scale > 0.f ? scale : 1.0f / sqrtf((float)head_dim);
    AttnCommon ac{};
    ac.counts = counts;
    ac.cu_q = cu_q;
    ac.query_lens = query_lens;
    ac.seq_lens = seq_lens;
    ac.block_table = block_table;
    ac.max_blocks = max_blocks_per_req;
    ac.page_size = page_size;
    ac.num_pages = num_pages;
    ac.num_q_heads = num_q_heads;
    ac.num_kv_heads = num_kv_heads;
    ac.group = group;
    ac.scale_log2 = sc * 1.4426950408889634f;
    ac.out = out;
    ac.part_o = part_o;
    ac.part_ml = part_ml;
    ac.dev_err = dev_err;
    ac.fused = fused ? 1 : 0;
    ac.k_new = k_new;
    ac.v_new = v_new;
    ac.slot_mapping = slot_mapping;
    ac.k_cache_w = k_cache;
    ac.v_cache_w = v_cache;

    const uint64_t D = (uint64_t)head_dim;
    const uint64_t rows_kv = (uint64_t)num_pages * (uint64_t)num_kv_heads;
    CUtensorMap tq, tk, tv, tkd, tvd;
    const uint32_t pb_chunk = page_size < 128 ? page_size : 128;
    if (!make_map(&tq, q, D, (uint64_t)num_q_heads, (uint64_t)num_tokens, D * 2, D * 2 * num_q_heads, 64, 1, 128) ||
        !make_map(&tk, k_cache, D, (uint64_t)page_size, rows_kv, D * 2, D * 2 * page_size, 64, pb_chunk, 1) ||
        !make_map(&tv, v_cache, D, (uint64_t)page_size, rows_kv, D * 2, D * 2 * page_size, 64, pb_chunk, 1))
        return CPSA_ERR_CUDA;
    // the new K/V rows, [T][Hkv][D]: 128-token boxes of one kv head (fused KV write)
    CUtensorMap tkn = tk, tvn = tv;
    if (fused && (!make_map(&tkn, k_new, D, (uint64_t)num_kv_heads, (uint64_t)num_tokens, D * 2,
                            D * 2 * num_kv_heads, 64, 1, 128) ||
                  !make_map(&tvn, v_new, D, (uint64_t)num_kv_heads, (uint64_t)num_tokens, D * 2,
                            D * 2 * num_kv_heads, 64, 1, 128)))
        return CPSA_ERR_CUDA;
    // decode: grouped, one box per page (16 rows, 8 at page 8) covering the item's
    // heads and all of head_dim; else one box per page-head block (at most 64 rows)
    const uint32_t pb_dec = page_size < kDecodeChunk ? page_size : kDecodeChunk;
    if (dec_heads > 1) {
        const uint32_t rows = page_size < 16 ? (uint32_t)page_size : 16u;
        if (!make_map_group(&tkd, k_cache, head_dim, page_size, num_kv_heads, num_pages, rows, dec_heads) ||
            !make_map_group(&tvd, v_cache, head_dim, page_size, num_kv_heads, num_pages, rows, dec_heads))
            return CPSA_ERR_CUDA;
    } else if (head_dim == 128) {
        if (!make_map4_halves(&tkd, k_cache, page_size, rows_kv, pb_dec) ||
            !make_map4_halves(&tvd, v_cache, page_size, rows_kv, pb_dec))
            return CPSA_ERR_CUDA;
    } else if (!make_map(&tkd, k_cache, D, (uint64_t)page_size, rows_kv, D * 2, D * 2 * page_size, 64, pb_dec, 1) ||
               !make_map(&tvd, v_cache, D, (uint64_t)page_size, rows_kv, D * 2, D * 2 * page_size, 64, pb_dec, 1)) {
        return CPSA_ERR_CUDA;
    }

    ChunkParams cp;
    static_cast<AttnCommon &>(cp) = ac;
    cp.pitems = pitems;
    cp.run_first = run_first;
    cp.flags = flags;
    cp.epoch = next_epoch();
    cp.self_plan = self_plan ? 1 : 0;
    cp.num_tokens = (int)num_tokens;
    // cuts need two pieces' partial rows per run (see the chunk kernel's self plan)
    const bool partials_fit = cap >= (int64_t)2 * pp.chunk_grid * kTileM * nq;
    cp.split_ok = max_kv_splits > 1 && partials_fit ? 1 : 0;
    cp.split_clamped = max_kv_splits > 1 && !partials_fit ? 1 : 0;
    // out, [T][Hq][D], in boxes of 64 columns x 1 head x 32 rows: the chunk
    // kernel's TMA stores of whole units' rows (head_dim 128 without the KV
    // write, whose cache writer holds the staging buffer) and of merged rows at
    // the end of a run; without the map the rows are stored directly
    CUtensorMap to = tq;
    cp.out_tma = head_dim == 128 && aligned16(out) &&
                         make_map(&to, out, D, (uint64_t)num_q_heads, (uint64_t)num_tokens, D * 2,
                                  D * 2 * num_q_heads, 64, 1, 32)
                     ? 1
                     : 0;
    // V below page 128: one box per page of one kv head, both column halves
    CUtensorMap tv4 = tv;
    if (head_dim == 128 && page_size < 128 && !make_map4_halves(&tv4, v_cache, page_size, rows_kv, page_size))
        return CPSA_ERR_CUDA;
    const int grid_c = single_decode ? 0 : pp.chunk_grid;   // one stream-K run per CTA
    if (grid_c > 0 &&
        launch_chunk_attn(cp, tq, tk, tv, tkn, tvn, to, tv4, head_dim, nq, grid_c, s, early && !self_plan) !=
            cudaSuccess)
        return CPSA_ERR_CUDA;
    mark(2, s);

    DecodeParams dp;
    static_cast<AttnCommon &>(dp) = ac;
    dp.ditems = ditems;
    dp.q = q;
    dp.k_cache_ptr = k_cache;
    dp.v_cache_ptr = v_cache;
    int grid_d = single_prefill ? 0 : (int)(L.max_ditems < sms ? L.max_ditems : sms);
    if (grid_d > 0 &&
        (dec_heads > 1 ? launch_decode_group(dp, tkd, tvd, head_dim, dec_heads, grid_d, s, early)
                       : launch_decode_attn(dp, tkd, tvd, head_dim, grid_d, s, early)) != cudaSuccess)
        return CPSA_ERR_CUDA;
    mark(3, s);

    // the combine kernel merges split decode rows (split prefill units are merged
    // in the chunk kernel): a single prefill request has none
    if (cap > 0 && !single_prefill) {
        CombineParams cb{counts, citems, part_o, part_ml, out, num_q_heads};
        const int grid_m = 4 * sms;
        if (grid_m > 0 && launch_combine(cb, head_dim, grid_m, s, early) != cudaSuccess)
            return CPSA_ERR_CUDA;
    }
    mark(4, s);
    return CPSA_OK;
}

}  // namespace

extern "C" {

int cpp_split_microbatch(const int32_t *query_lens, int num_reqs, float balance_threshold, int32_t length_threshold,
                         int32_t *out3, void *stream)
{
    if (num_reqs < 0 || num_reqs >= (1 << 24))
        return CPSA_ERR_BAD_SHAPE;
    if (!out3 || (num_reqs > 0 && !query_lens))
        return CPSA_ERR_NULL_ARG;
    cudaError_t e = launch_split_microbatch(query_lens, num_reqs, balance_threshold, length_threshold, out3,
                                            (cudaStream_t)stream);
    return e == cudaSuccess ? CPSA_OK : CPSA_ERR_CUDA;
}

int cpp_selftest_exp2(const float *x, float *out_poly, float *out_hw, int64_t n, void *stream)
{
    if (n < 0)
        return CPSA_ERR_BAD_SHAPE;
    if (n > 0 && (!x || !out_poly || !out_hw))
        return CPSA_ERR_NULL_ARG;
    return launch_exp2_selftest(x, out_poly, out_hw, n, (cudaStream_t)stream) == cudaSuccess ? CPSA_OK
                                                                                             : CPSA_ERR_CUDA;
}

int cpp_selftest_wait_timeout(int64_t limit_ns, uint32_t *dev_err, int32_t *out3, void *stream)
{
    if (limit_ns < 1000 || limit_ns > 100000000)
        return CPSA_ERR_BAD_SHAPE;
    if (!dev_err || !out3)
        return CPSA_ERR_NULL_ARG;
    return launch_wait_selftest((uint64_t)limit_ns, dev_err, out3, (cudaStream_t)stream) == cudaSuccess
               ? CPSA_OK
               : CPSA_ERR_CUDA;
}

int cpp_read_device_error(uint32_t *dev_err, uint32_t *host_flags, int clear, void *stream)
{
    if (!dev_err || !host_flags)
        return CPSA_ERR_NULL_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemcpyAsync(host_flags, dev_err, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return CPSA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return CPSA_ERR_CUDA;
    if (clear && cudaMemsetAsync(dev_err, 0, sizeof(uint32_t), s) != cudaSuccess)
        return CPSA_ERR_CUDA;
    return CPSA_OK;
}

int cpp_get_device_error(const uint32_t *dev_err, uint32_t *host_flags, void *stream)
{
    return cpp_read_device_error(const_cast<uint32_t *>(dev_err), host_flags, 0, stream);
}

}  // extern "C"
