/*
 * cpsa.h -- C ABI of libcpsa.so: chunked-prefill attention over a paged KV cache
 * for NVIDIA GB300 (sm_103a).
 *
 * Sources of the operations (web pages, by title and section):
 *   [CP]  "vLLM Chunked-Prefills" article (Sarathi-Serve chunked prefill), section
 *         3.1 (chunks of a long prompt, each caching its KV; decode rows first in
 *         the token budget) and 3.2.1 (chunked attention: a chunk's queries against
 *         the cached history keys concatenated with its own keys, softmax, values).
 *   [DS]  Ascend "dual-stream parallel for Qwen3 dense" article, section 3.1:
 *         attn_metadata (num_actual_tokens, slot_mapping, seq_lens, query_lens,
 *         block_table) and the choice of the micro-batch split point.
 *   [CPP] vllm-ascend design page "Dynamic Chunked Pipeline Parallel (CPP)":
 *         quadratic latency model, chunk-size solver, online calibration.
 *
 * Conventions for every entry point:
 *   - bf16 tensors are passed as void* and hold IEEE bfloat16 values.
 *   - Device pointers belong to the caller; the library never allocates device
 *     memory, keeps no device state between calls, and never synchronises the
 *     stream except in cpp_read_device_error.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream); all work is
 *     enqueued on it in order.
 *   - Return value: CPSA_OK, or a negative CPSA_ERR_* detected on the host, in
 *     which case nothing was launched.
 *   - Data-dependent problems found on the device (an index out of range, a bad
 *     length) set bits in the caller's 32-bit device word `dev_err` with
 *     atomicOr; the offending item is skipped and no kernel traps. Read and
 *     clear the word with cpp_read_device_error.
 *
 * Layouts (row-major, innermost last):
 *   q            [num_tokens][num_q_heads][head_dim]      bf16, token-major
 *   k, v         [num_tokens][num_kv_heads][head_dim]     bf16, the new tokens' K/V
 *   k/v_cache    [num_pages][num_kv_heads][page_size][head_dim] bf16
 *   out          [num_tokens][num_q_heads][head_dim]      bf16
 *   slot_mapping [num_tokens] int64: slot = page * page_size + offset; < 0 = padding
 *   block_table  [num_reqs][max_blocks_per_req] int32 page indices; entries past a
 *                request's last page are never read (any value, e.g. -1)
 *   query_lens, seq_lens [num_reqs] int32: seq_len counts the cached history plus
 *                the request's new tokens; the new tokens are the last query_len
 *                positions and sit contiguously in q in request order.
 * Supported shapes: head_dim 64 or 128; num_q_heads a multiple of num_kv_heads
 * with at most 16 q heads per kv head; page_size a power of two in [8, 256];
 * all base pointers 16-byte aligned.
 */
#ifndef CPSA_H
#define CPSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- host status codes ---------------------------------------------------- */
#define CPSA_OK 0
#define CPSA_ERR_NULL_ARG (-1)            /* a required pointer is NULL */
#define CPSA_ERR_BAD_SHAPE (-2)           /* a size or count is negative / inconsistent */
#define CPSA_ERR_MISALIGNED (-3)          /* a base pointer is not 16-byte aligned */
#define CPSA_ERR_UNSUPPORTED (-4)         /* head_dim, head grouping or page_size not supported */
#define CPSA_ERR_WORKSPACE_TOO_SMALL (-5) /* workspace below cpp_attn_workspace_min_bytes */
#define CPSA_ERR_CUDA (-6)                /* a CUDA runtime call or launch failed */
#define CPSA_ERR_NO_DEVICE (-7)           /* no usable sm_103 device is current */
#define CPSA_ERR_SCRATCH_TOO_SMALL (-8)   /* batch needs more than the built-in scratch area */
#define CPSA_ERR_SCRATCH_UNAVAILABLE (-9) /* the built-in scratch area could not be reserved in this context */

/* ---- device error flags (bits of *dev_err) --------------------------------- */
#define CPSA_DEV_SLOT_OUT_OF_RANGE 0x01u  /* slot >= num_pages * page_size: token skipped */
#define CPSA_DEV_PAGE_OUT_OF_RANGE 0x02u  /* block_table entry outside [0, num_pages): tile skipped */
#define CPSA_DEV_SEQ_LT_QUERY 0x04u       /* seq_len < query_len or query_len < 0: request skipped */
#define CPSA_DEV_TOKENS_MISMATCH 0x08u    /* sum(query_lens) != num_tokens: nothing computed */
#define CPSA_DEV_SEQ_GT_TABLE 0x10u       /* seq_len > max_blocks_per_req * page_size: request skipped */
#define CPSA_DEV_SPLITS_CLAMPED 0x20u     /* info: partials did not fit the workspace, one KV split used */
#define CPSA_DEV_WAIT_TIMEOUT 0x40u       /* an on-chip wait hit its limit; outputs of this call invalid */
#define CPSA_DEV_PLAN_OVERFLOW 0x80u      /* a self-planned chunk-kernel run held more pieces than it can keep */

/*
 * Write the new tokens' K and V into their cache slots ([DS] section 3.1,
 * slot_mapping: "map each token position to its slot").
 *
 * For each token t with s = slot_mapping[t] >= 0:
 *   k_cache[s / page_size][h][s % page_size][:] = k[t][h][:]  for every kv head h,
 *   and the same for v. A bit copy; other cache bytes are untouched.
 * Tokens with s < 0 are padding and skipped; s >= num_pages * page_size sets
 * CPSA_DEV_SLOT_OUT_OF_RANGE and the token is skipped. Duplicate slots within
 * one call leave an unspecified one of the writers' values.
 * Run it before cpp_chunked_prefill_attn on the same stream: attention reads the
 * chunk's own K/V from the cache.
 */
int cpp_kv_cache_write(const void *k, const void *v, const int64_t *slot_mapping,
                       int64_t num_tokens, int num_kv_heads, int head_dim, int page_size,
                       int64_t num_pages, void *k_cache, void *v_cache, uint32_t *dev_err,
                       void *stream);

/*
 * Workspace for cpp_chunked_prefill_attn, in bytes.
 *
 * cpp_attn_workspace_bytes is the size that lets every row use up to
 * max_kv_splits KV splits (partial results are stored for every token and head
 * in the worst case); cpp_attn_workspace_min_bytes is the metadata part alone.
 * Any size in between is accepted: when a call's partial results do not fit,
 * the call runs every row with one split and sets CPSA_DEV_SPLITS_CLAMPED.
 * Returns 0 for invalid arguments.
 */
size_t cpp_attn_workspace_bytes(int num_reqs, int64_t num_tokens, int num_q_heads,
                                int num_kv_heads, int head_dim, int max_kv_splits);
size_t cpp_attn_workspace_min_bytes(int num_reqs, int64_t num_tokens, int num_q_heads,
                                    int num_kv_heads, int head_dim, int max_kv_splits);

/*
 * Causal chunked-prefill attention over the paged cache, mixed with decode rows
 * ([CP] section 3.2.1 for the computation, [DS] section 3.1 for the metadata).
 *
 * For request r with q_r = query_lens[r], s_r = seq_lens[r], h_r = s_r - q_r, new
 * token i (0 <= i < q_r, global row t = sum_{r'<r} q_r' + i) and q head h:
 *   keys j = 0 .. h_r + i of kv head h / (num_q_heads / num_kv_heads), key j at
 *   k_cache[block_table[r][j / page_size]][kvh][j % page_size];
 *   out[t][h] = sum_j softmax_j(scale * q[t][h] . k_j) * v_j      (bf16 result)
 * scale <= 0 selects 1 / sqrt(head_dim). A request with q_r = 1 is a decode row
 * and takes the split-KV decode kernel; q_r >= 2 takes the tensor-core chunk
 * kernel; q_r = 0 contributes nothing. Arithmetic: bf16 inputs, fp32
 * accumulation and softmax, probabilities rounded to bf16 before P.V.
 *
 * max_kv_splits (>= 1) caps the number of KV splits of a decode row; that count
 * depends only on the row's own seq_len and max_kv_splits. Prefill rows are split
 * stream-K style: the KV tiles of all prefill units of the batch (128 query rows
 * x kv head x q-head pair) are laid end to end and cut into equal runs, one per
 * CTA of the chunk kernel (unless every unit is at least a run long and the
 * longest within a few tiles of it: then units stay whole, one per CTA), and a
 * unit cut by a run boundary is merged inside the chunk kernel from partial
 * results (per piece O / l in bf16 with fp32 row max and sum; split decode rows
 * by the combine kernel from fp32 partials, launched only when the batch holds
 * decode rows). Where the cuts fall depends on the whole batch, so a prefill
 * row's last-bit rounding (not its value) can depend on the other requests; it
 * does not depend on timing.
 * max_kv_splits = 1 turns off both kinds of split.
 * A batch of one prefill request (num_reqs == 1, num_tokens >= 2) of at most
 * about 6.6k tokens at 32/8 heads (while every CTA's run fits 56 pieces)
 * launches the chunk kernel alone: its CTAs compute their own runs, with the
 * same units and cuts.
 * workspace: device memory of at least cpp_attn_workspace_min_bytes(...) with
 * the same (num_reqs, num_tokens, heads, head_dim, max_kv_splits); it is
 * scratch, overwritten by each call; calls that share it must be stream-ordered.
 * No call needs the workspace cleared: the merge counters a call uses are
 * cleared by the call itself as each split unit is merged, and are tagged with
 * the call's epoch (a per-call number) so that counts left by a call that ended
 * with a device error read as zero in the next call.
 * CUDA graphs: the call may be captured on `stream` and replayed; a replay
 * keeps the sizes, pointers and epoch of the capture and reads the current
 * contents of the buffers. After a replay that reported a device error, clear
 * the workspace (or call once outside the graph) before the next replay.
 */
int cpp_chunked_prefill_attn(const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *query_lens, const int32_t *seq_lens,
                             const int32_t *block_table, int num_reqs, int64_t num_tokens,
                             int max_blocks_per_req, int num_q_heads, int num_kv_heads,
                             int head_dim, int page_size, int64_t num_pages, float scale,
                             int max_kv_splits, void *out, void *workspace,
                             size_t workspace_bytes, uint32_t *dev_err, void *stream);

/*
 * cpp_chunked_prefill_attn with timing marks: when `events` is not NULL it
 * points to 5 cudaEvent_t handles (any may be NULL) recorded on `stream`:
 * [0] before the plan kernel (when one runs), [1] before the chunk kernel, [2] after it,
 * [3] after the decode kernel, [4] after the combine kernel (kernels that a
 * batch does not need are not launched; their marks follow the previous one).
 * For profiling harnesses; the computation is identical, its kernels launched
 * in plain stream order. Under stream capture the marks are recorded as
 * external events (cudaEventRecordExternal), so a call captured in a CUDA graph
 * records them as event nodes at every replay and their timings can be read
 * afterwards.
 */
int cpp_chunked_prefill_attn_events(const void *q, const void *k_cache, const void *v_cache,
                                    const int32_t *query_lens, const int32_t *seq_lens,
                                    const int32_t *block_table, int num_reqs, int64_t num_tokens,
                                    int max_blocks_per_req, int num_q_heads, int num_kv_heads,
                                    int head_dim, int page_size, int64_t num_pages, float scale,
                                    int max_kv_splits, void *out, void *workspace,
                                    size_t workspace_bytes, uint32_t *dev_err, void *stream,
                                    void *const *events);

/*
 * The KV write fused into the attention: cpp_kv_cache_write followed by
 * cpp_chunked_prefill_attn in one call, with no separate write kernel and no
 * re-read of the new rows from the cache ([DS] section 3.1 for the write and
 * the metadata, [CP] section 3.2.1 for the attention, whose chunk attends to
 * its own keys alongside the cached history).
 *
 * k, v: bf16 [num_tokens][num_kv_heads][head_dim], contiguous, 16-byte aligned
 * (the layout of cpp_kv_cache_write); slot_mapping: int64 [num_tokens]; both
 * caches are written. Every other argument, the workspace and the device flags
 * are those of cpp_chunked_prefill_attn.
 *
 * Attention reads the history keys (positions < h_r) from the cache through
 * block_table and the new tokens' keys and values straight from k and v, so
 * its result equals the two-call sequence whenever token i of request r is
 * placed at slot block_table[r][(h_r + i) / page_size] * page_size + (h_r + i) %
 * page_size, the usual case. Each new row is also stored, once and bit for bit,
 * to k_cache / v_cache at slot_mapping[t] with the rules of cpp_kv_cache_write
 * (s < 0 skipped, s past the cache flagged with CPSA_DEV_SLOT_OUT_OF_RANGE and
 * skipped). Rows of requests that fail validation (CPSA_DEV_SEQ_LT_QUERY,
 * CPSA_DEV_SEQ_GT_TABLE, CPSA_DEV_TOKENS_MISMATCH) are neither attended nor
 * stored. The stores of a call become visible to later stream-ordered work; no
 * part of the same call reads them. With every h_r a multiple of 128 the output
 * is bit-identical to the two-call sequence; otherwise the chunk's keys are
 * tiled from h_r rather than from a multiple of 128 and the output agrees to
 * the attention's rounding.
 */
int cpp_chunked_prefill_attn_write_kv(const void *q, const void *k, const void *v,
                                      const int64_t *slot_mapping, void *k_cache, void *v_cache,
                                      const int32_t *query_lens, const int32_t *seq_lens,
                                      const int32_t *block_table, int num_reqs, int64_t num_tokens,
                                      int max_blocks_per_req, int num_q_heads, int num_kv_heads,
                                      int head_dim, int page_size, int64_t num_pages, float scale,
                                      int max_kv_splits, void *out, void *workspace,
                                      size_t workspace_bytes, uint32_t *dev_err, void *stream);

/* cpp_chunked_prefill_attn_write_kv with the 5 timing events of
 * cpp_chunked_prefill_attn_events (same positions, same plain stream order). */
int cpp_chunked_prefill_attn_write_kv_events(const void *q, const void *k, const void *v,
                                             const int64_t *slot_mapping, void *k_cache,
                                             void *v_cache, const int32_t *query_lens,
                                             const int32_t *seq_lens, const int32_t *block_table,
                                             int num_reqs, int64_t num_tokens,
                                             int max_blocks_per_req, int num_q_heads,
                                             int num_kv_heads, int head_dim, int page_size,
                                             int64_t num_pages, float scale, int max_kv_splits,
                                             void *out, void *workspace, size_t workspace_bytes,
                                             uint32_t *dev_err, void *stream, void *const *events);

/*
 * cpp_chunked_prefill_attn for callers that cannot allocate device memory.
 * (The pages have no counterpart of this call; it exists for library users.)
 *
 * Who needs it: code that runs inside a host application that owns all device
 * memory and forbids allocation on its serving path, or C callers with no
 * allocator of their own. Instead of a caller workspace it uses a scratch area
 * the library owns: a fixed array of CPSA_NOALLOC_SCRATCH_BYTES in device
 * global memory, kept until the process exits. The call itself allocates
 * nothing: the array is reserved when the library's device code is loaded into
 * a CUDA context, which with CUDA's default lazy module loading is the first
 * call of this function in that context (or any earlier call of the library
 * that loads the same code). A host that claims all device memory up front
 * should therefore make one warm-up call at initialisation; when the array
 * cannot be reserved the call returns CPSA_ERR_SCRATCH_UNAVAILABLE.
 *
 * Same arguments, results and device flags as cpp_chunked_prefill_attn, minus
 * the workspace. Returns CPSA_ERR_SCRATCH_TOO_SMALL when the batch's work lists
 * (cpp_attn_workspace_min_bytes) exceed the scratch area; when only the split
 * partials do not fit, every row runs with one KV split and
 * CPSA_DEV_SPLITS_CLAMPED is set, as with a small workspace.
 * The array's device address belongs to a CUDA context: the first call in each
 * context (the calling thread's current one; the device's primary context for
 * runtime-API callers) looks it up and caches it under the context's unique ID,
 * so contexts created through the driver API, and a primary context rebuilt
 * after cudaDeviceReset, each get their own lookup. Make that first call in a
 * context before any stream capture. All calls in a context share the one
 * area and find it holding the previous call's data (the call rewrites
 * everything it reads, the merge counters included), so calls whose execution
 * overlaps on the GPU -- on different streams, or from different host threads
 * -- race and must be ordered by the caller.
 */
#define CPSA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int cpp_chunked_prefill_attn_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                     const int32_t *query_lens, const int32_t *seq_lens,
                                     const int32_t *block_table, int num_reqs, int64_t num_tokens,
                                     int max_blocks_per_req, int num_q_heads, int num_kv_heads,
                                     int head_dim, int page_size, int64_t num_pages, float scale,
                                     int max_kv_splits, void *out, uint32_t *dev_err, void *stream);

/*
 * The device address of cpp_chunked_prefill_attn_noalloc's scratch area in the
 * calling thread's current CUDA context (the device's primary context when no
 * context is current), written to *addr: the same lookup, and the same
 * per-context cache, as the first attention call in that context (so it also
 * reserves the area, and can serve as the warm-up call). Launches nothing.
 * Returns CPSA_OK, CPSA_ERR_NO_DEVICE, CPSA_ERR_SCRATCH_UNAVAILABLE or
 * CPSA_ERR_CUDA; *addr is left unchanged on an error.
 */
int cpp_noalloc_scratch_address(void **addr);

/*
 * Balanced micro-batch split point ([DS] section 3.1, "advanced method").
 *
 * total = sum(query_lens); best = total / 2 (integer); over request boundaries
 * k = 1 .. num_reqs-1 with cum_k = sum_{r<k} query_lens[r], pick the k nearest to
 * best (smallest k on ties); n1 = cum_k, n2 = total - n1;
 * use_two = |n1 - n2| / min(n1, n2) <= balance_threshold and
 *           min(n1, n2) >= length_threshold (and min > 0).
 * Writes out3[0] = k (batch split), out3[1] = n1 (token split), out3[2] = use_two
 * into DEVICE memory; num_reqs < 2 gives (0, 0, 0). query_lens must be >= 0.
 */
int cpp_split_microbatch(const int32_t *query_lens, int num_reqs, float balance_threshold,
                         int32_t length_threshold, int32_t *out3, void *stream);

/*
 * Copy the device error word to *host_flags (synchronises `stream`), and reset
 * it to zero when clear != 0.
 */
int cpp_read_device_error(uint32_t *dev_err, uint32_t *host_flags, int clear, void *stream);

/*
 * Copy the device error word to *host_flags without resetting it (synchronises
 * `stream`): cpp_read_device_error with clear = 0, under the name the contract
 * of this boundary gives the read.
 */
int cpp_get_device_error(const uint32_t *dev_err, uint32_t *host_flags, void *stream);

/*
 * Host-side chunk planner ([CPP] "runtime phase: dynamic prediction").
 *
 * Latency model f(l) = a l^2 + b l + c; target T = f(base_chunk_size) - f(0).
 * From prefix L, the next chunk x solves f(L + x) - f(L) = T (positive root,
 * evaluated as 2T / ((2aL+b) + sqrt((2aL+b)^2 + 4aT)); a <= 0 gives T / b, and
 * b <= 0 as well gives base_chunk_size); then x is blended with base by
 * smooth_factor (x_s = s x + (1 - s) base), rounded down to a multiple of
 * page_size (relative slack 1e-9) with a minimum of min_chunk, capped at
 * max_model_len - L and max_num_scheduled_tokens (values <= 0 mean no cap), and
 * at the remaining prompt. Writes up to max_chunks sizes; *n_chunks gets the
 * count needed. Returns CPSA_ERR_BAD_SHAPE if chunks was too short.
 */
int cpp_plan_chunk_sizes(double a, double b, double c, int64_t prompt_len,
                         int64_t base_chunk_size, int page_size, int64_t min_chunk,
                         int64_t max_model_len, int64_t max_num_scheduled_tokens,
                         double smooth_factor, int64_t *chunks, int64_t max_chunks,
                         int64_t *n_chunks);

/*
 * Least-squares fits of the latency models ([CPP] "startup phase: profiling" and
 * "online calibration"). n samples; coef[3] = (a, b, c).
 *   quadratic: f(l) = a l^2 + b l + c, samples (l[i], t[i]);
 *   two-variable: f(C, H) = a C (C + H) + b (C + H) + c, with per-sample
 *   features x0 = sum C (C + H), x1 = sum (C + H), x2 = number of chunks.
 * Returns CPSA_ERR_BAD_SHAPE when n < 3 or the system is singular.
 */
int cpp_fit_latency_quadratic(const double *l, const double *t, int n, double *coef);
int cpp_fit_latency_two_var(const double *x0, const double *x1, const double *x2,
                            const double *t, int n, double *coef);

/*
 * Online chunk-size controller ([CPP] "online calibration"): the planner above,
 * but fed back with the measured time of every batch it sized.
 *
 * Until min_points batches are recorded it sizes chunks with the startup model
 * (a, b, c of f(l), exactly as cpp_plan_chunk_sizes). Each recorded batch adds
 * the features [sum C (C + H), sum (C + H), N] of its N chunks (size C, history
 * H) and its time; from min_points batches on, (a, b, c) of the two-variable
 * model f(C, H) = a C (C + H) + b (C + H) + c are refitted by least squares over
 * the last `window` batches (the page gives 5 to 30 points), and the next chunk
 * at history H solves f(C, H) - f(0, H) = T, i.e. a C^2 + (aH + b) C - T = 0,
 * with T = f(base, 0) - f(0, 0) = a base^2 + b base from the current model;
 * smoothing, page alignment, minimum and caps as in cpp_plan_chunk_sizes, and
 * at most `remaining` tokens. A singular refit keeps the previous model.
 *
 * The handle is host memory owned by the library: create it once, destroy it
 * with cpp_online_destroy. Not thread-safe; every call is host-only.
 * cpp_online_create returns NULL on invalid arguments (base, page_size or
 * min_chunk < 1, window < 3, min_points < 3 or > window).
 */
typedef struct cpsa_online cpsa_online;
cpsa_online *cpp_online_create(double a, double b, double c, int64_t base_chunk_size, int page_size,
                               int64_t min_chunk, int64_t max_model_len, int64_t max_num_scheduled_tokens,
                               double smooth_factor, int window, int min_points);
void cpp_online_destroy(cpsa_online *handle);
int cpp_online_next_chunk(const cpsa_online *handle, int64_t history, int64_t remaining, int64_t *chunk);
int cpp_online_record(cpsa_online *handle, const int64_t *chunks, const int64_t *histories, int n_chunks,
                      double time_ms);
/* coef[3] = current (a, b, c); *n_samples batches recorded; *calibrated = 1 once refitted */
int cpp_online_model(const cpsa_online *handle, double *coef, int *n_samples, int *calibrated);

/*
 * Token-budget batch builder with page allocation ([CP] section 3: the
 * scheduling cycle; section 3.2.2: chunk-size strategies). Host only.
 *
 * Each step builds one batch under token_budget tokens: decode rows first (one
 * token each, admission order), then prompts already started, each taking
 * min(remaining prompt, budget left) tokens, then waiting requests in arrival
 * order while budget is left. A prefill chunk is also capped by
 * chunk_caps[min(i, n_caps - 1)] for the prompt's i-th chunk (n_caps = 0: no
 * cap; {2048, 1024, 512} is the progressive strategy) and, when it is not the
 * prompt's last, rounded down to a multiple of tile_align (0: none).
 * Pages come from a free list (page_order, or 0 .. num_pages - 1 when NULL),
 * taken from the front as a request's sequence grows and returned to the back
 * when it finishes (prompt prefilled and max_new_tokens decode rows run). A
 * decode row or started prompt whose tokens do not fit in the free pages is
 * skipped for the step; admission stops at the first waiting request that does
 * not fit. A step that schedules nothing while requests remain means the pool
 * is too small: the caller must stop.
 *
 * cpp_sched_step writes the batch for cpp_kv_cache_write and
 * cpp_chunked_prefill_attn into HOST arrays: req_ids[B], query_lens[B],
 * seq_lens[B] (history + this step's tokens), block_table[B][max_blocks]
 * (-1 padded), slot_mapping[T] (positions seq_len - query_len .. seq_len - 1 of
 * each request, batch order). It fails with CPSA_ERR_BAD_SHAPE, changing
 * nothing, when max_reqs, max_tokens or max_blocks is too small, or when the
 * previous step was not committed. cpp_sched_commit applies the last step's
 * progress (call it once the step's kernels are enqueued). The handle is host
 * memory owned by the library; not thread-safe.
 */
typedef struct cpsa_sched cpsa_sched;
cpsa_sched *cpp_sched_create(int64_t token_budget, int page_size, int64_t num_pages, const int32_t *page_order,
                             const int64_t *chunk_caps, int n_caps, int tile_align);
void cpp_sched_destroy(cpsa_sched *handle);
int cpp_sched_add_request(cpsa_sched *handle, int64_t id, int64_t prompt_len, int64_t max_new_tokens);
int cpp_sched_step(cpsa_sched *handle, int max_reqs, int64_t max_tokens, int max_blocks, int64_t *req_ids,
                   int32_t *query_lens, int32_t *seq_lens, int32_t *block_table, int64_t *slot_mapping,
                   int *n_reqs, int64_t *n_tokens);
int cpp_sched_commit(cpsa_sched *handle);
int cpp_sched_stats(const cpsa_sched *handle, int64_t *waiting, int64_t *running, int64_t *finished,
                    int64_t *free_pages);

/*
 * Self-test of the attention kernels' two base-2 exponentials on n device floats:
 * out_poly[i] = the FMA-pipe polynomial path (x clamped to [-125, 127]; range
 * reduction to f in [-1/2, 1/2] plus a degree-3 minimax polynomial, relative
 * error 7.5e-5), out_hw[i] = the hardware ex2.approx. Stream-ordered.
 */
int cpp_selftest_exp2(const float *x, float *out_poly, float *out_hw, int64_t n, void *stream);

/*
 * Self-test of failure detection (no counterpart in the pages; the kernels'
 * bounded waits). One CTA: warp 0 waits on an mbarrier that nothing arrives at,
 * with a limit of limit_ns (1 us .. 100 ms, else CPSA_ERR_BAD_SHAPE); when it
 * runs out it sets the CTA's abort flag, the way a stalled copy or MMA would in
 * the attention kernels. Warp 1 waits on a second such barrier with the
 * kernels' standard one-second limit and must leave as soon as it sees the
 * abort flag. CPSA_DEV_WAIT_TIMEOUT is then set in *dev_err. out3 (device
 * int32[3]): warp 0's wait succeeded (1) or gave up (0); the same for warp 1;
 * microseconds warp 1 waited. Stream-ordered; the kernel always ends (within
 * limit_ns plus the abort poll), and leaves the context usable.
 */
int cpp_selftest_wait_timeout(int64_t limit_ns, uint32_t *dev_err, int32_t *out3, void *stream);

/* Human-readable name of a status code. */
const char *cpp_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* CPSA_H */
