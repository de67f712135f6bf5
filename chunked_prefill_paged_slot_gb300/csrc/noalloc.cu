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

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = CPSA_NOALLOC_SCRATCH_BYTES;

// The library's scratch area. Its host-side name is only a handle for
// cudaGetSymbolAddress, never a device address.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch area on the current device, looked up once per
// device (with that device current) and cached.
int scratch_address(void **addr)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return CPSA_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return CPSA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
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
