// noalloc.cu -- cpp_chunked_prefill_attn_noalloc: the attention call for
// callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: a plugin loaded into
// a host application that owns every byte of device memory and forbids
// allocation on its serving path, or plain C code that has no allocator of its
// own next to a framework's caching allocator (a cudaMalloc there would also
// synchronise the device in the middle of a step). For them this entry point
// uses a scratch area that the library itself owns: a fixed array in device
// global memory, reserved when the library's device code is loaded on a GPU and
// kept until the process exits. The computation is the one of
// cpp_chunked_prefill_attn, fed that array as its workspace.
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = CPSA_NOALLOC_SCRATCH_BYTES;

// The library's scratch area. Its host-side name is only a handle for
// cudaGetSymbolAddress, never a device address.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// A __device__ array has one address per CUDA context, not per device: a host
// that drives contexts of its own through the driver API sees a different
// address for each, and a primary context rebuilt after cudaDeviceReset may
// hold the array elsewhere. So the address is cached per context, under the
// context's unique ID (cuCtxGetId: never reused within a process, unlike a
// context handle).
constexpr int kMaxContexts = 64;
std::mutex g_scratch_mutex;
unsigned long long g_ctx_id[kMaxContexts] = {};
void *g_ctx_addr[kMaxContexts] = {};
int g_n_ctx = 0;

PFN_cuCtxGetCurrent_v4000 g_get_current = nullptr;
PFN_cuCtxGetId_v12000 g_get_id = nullptr;

bool driver_fns()
{
    if (g_get_current && g_get_id)
        return true;
    void *f0 = nullptr, *f1 = nullptr;
    cudaDriverEntryPointQueryResult q0, q1;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f0, 4000, cudaEnableDefault, &q0) != cudaSuccess ||
        q0 != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess)
        return false;
    g_get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f0);
    g_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f1);
    return true;
}

// Device address of the scratch area in the calling thread's current context,
// looked up once per context (that lookup loads the library's device code into
// the context if it is not loaded yet, which is when the array is reserved).
int scratch_address(void **addr)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0)
        return CPSA_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!driver_fns())
        return CPSA_ERR_CUDA;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    void *p = nullptr;
    if (g_get_current(&ctx) != CUDA_SUCCESS)
        return CPSA_ERR_NO_DEVICE;
    if (ctx) {
        if (g_get_id(ctx, &id) != CUDA_SUCCESS)
            return CPSA_ERR_NO_DEVICE;
        for (int i = 0; i < g_n_ctx; ++i)
            if (g_ctx_id[i] == id) {
                *addr = g_ctx_addr[i];
                return CPSA_OK;
            }
    }
    // Not cached (or no context current yet: the runtime makes the device's
    // primary context current here, on this lookup).
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        (void)cudaGetLastError();   // the failure is reported by the status, not left behind
        return CPSA_ERR_SCRATCH_UNAVAILABLE;
    }
    if (!ctx && (g_get_current(&ctx) != CUDA_SUCCESS || !ctx || g_get_id(ctx, &id) != CUDA_SUCCESS))
        return CPSA_ERR_NO_DEVICE;
    // a full table overwrites an entry (that context's next call looks up again)
    const int slot = g_n_ctx < kMaxContexts ? g_n_ctx++ : (int)(id % kMaxContexts);
    g_ctx_id[slot] = id;
    g_ctx_addr[slot] = p;
    *addr = p;
    return CPSA_OK;
}

}  // namespace

extern "C" int cpp_chunked_prefill_attn_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                                const int32_t *query_lens, const int32_t *seq_lens,
                                                const int32_t *block_table, int num_reqs, int64_t num_tokens,
                                                int max_blocks_per_req, int num_q_heads, int num_kv_heads,
                                                int head_dim, int page_size, int64_t num_pages, float scale,
                                                int max_kv_splits, void *out, uint32_t *dev_err, void *stream)
{
    // The batch's work lists must fit; split partials use whatever room is left
    // (when they do not fit, every row runs with one split).
    const size_t need = cpp_attn_workspace_min_bytes(num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim,
                                                     max_kv_splits);
    if (need > kScratchBytes)
        return CPSA_ERR_SCRATCH_TOO_SMALL;
    void *scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != CPSA_OK)
        return st;
    // The plan kernel rewrites every field of the scratch that the later kernels
    // read (counts, offsets, item lists, partial rows), so nothing is cleared here.
    return cpp_chunked_prefill_attn(q, k_cache, v_cache, query_lens, seq_lens, block_table, num_reqs, num_tokens,
                                    max_blocks_per_req, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                                    scale, max_kv_splits, out, scratch, kScratchBytes, dev_err, stream);
}

extern "C" int cpp_noalloc_scratch_address(void **addr)
{
    if (!addr)
        return CPSA_ERR_CUDA;
    void *p = nullptr;
    const int st = scratch_address(&p);
    if (st == CPSA_OK)
        *addr = p;
    return st;
}
