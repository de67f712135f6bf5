// scheduler.cpp -- host-side token-budget batch builder with page allocation,
// the loop that feeds the attention kernels step after step.
//
// Batch building follows the scheduling cycle of the "vLLM Chunked-Prefills"
// article (section 3, non-blocking scheduling with a token budget): decode rows
// first, one token each while the budget lasts; then the requests whose prompt
// is partly prefilled, each taking min(remaining prompt, budget); then new
// requests in arrival order while budget is left. Its chunk-size strategies
// (section 3.2.2) are options of the same cycle: a per-chunk cap list (the
// progressive [2048, 1024, 512] strategy: chunk i of a prompt is capped by
// caps[min(i, n - 1)]) and tile alignment (a chunk that is not the last of its
// prompt is rounded down to a multiple of tile_align).
//
// Pages: each request holds the pages of its sequence in order; a step
// allocates the pages its new tokens need from a free list (taken from the
// front, returned to the back when a request finishes), so block_table row r
// lists request r's pages and slot = page * page_size + position % page_size.
// A decode row or started prompt whose new tokens do not fit in the free pages
// is left out of the step; admission of new requests stops at the first one
// whose first chunk does not fit. A step that schedules nothing while requests
// remain means the pool is too small for them: the caller must stop.
#include <stdint.h>

#include <deque>
#include <new>
#include <vector>

#include "../../include/cpsa.h"

namespace {

struct Request {
    int64_t id, prompt_len, max_new;
    int64_t prefilled = 0;     // prompt tokens whose K/V is in the cache
    int64_t decoded = 0;       // decode rows run
    int64_t chunks = 0;        // prefill chunks taken so far
    std::vector<int32_t> pages;
    int64_t seq() const { return prefilled + decoded; }
};

struct Entry {
    int idx;        // index into running
    int64_t tokens;
    bool decode;
};

}  // namespace

struct cpsa_sched {
    int64_t budget;
    int page_size;
    std::vector<int64_t> caps;
    int tile_align;
    std::deque<int32_t> free_pages;
    std::deque<Request> waiting;          // not yet admitted
    std::vector<Request> running;         // admitted, in admission order
    std::vector<Entry> last;              // the batch of the last step, until commit
    bool pending = false;
    int64_t finished = 0;
};

namespace {

int64_t chunk_cap(const cpsa_sched *h, int64_t chunk_index)
{
    if (h->caps.empty())
        return INT64_MAX;
    const size_t i = chunk_index < (int64_t)h->caps.size() ? (size_t)chunk_index : h->caps.size() - 1;
    return h->caps[i];
}

// Tokens of the next prefill chunk of r under the budget, caps and alignment.
int64_t prefill_chunk(const cpsa_sched *h, const Request &r, int64_t budget)
{
    const int64_t rem = r.prompt_len - r.prefilled;
    int64_t c = rem < budget ? rem : budget;
    const int64_t cap = chunk_cap(h, r.chunks);
    if (c > cap)
        c = cap;
    if (c < rem && h->tile_align > 0)
        c -= c % h->tile_align;
    return c > 0 ? c : 0;
}

int64_t pages_needed(const cpsa_sched *h, const Request &r, int64_t tokens)
{
    const int64_t s = r.seq() + tokens;
    const int64_t need = (s + h->page_size - 1) / h->page_size;
    return need > (int64_t)r.pages.size() ? need - (int64_t)r.pages.size() : 0;
}

}  // namespace

extern "C" {

cpsa_sched *cpp_sched_create(int64_t token_budget, int page_size, int64_t num_pages, const int32_t *page_order,
                             const int64_t *chunk_caps, int n_caps, int tile_align)
{
    if (token_budget < 1 || page_size < 1 || num_pages < 0 || n_caps < 0 || (n_caps > 0 && !chunk_caps) ||
        tile_align < 0 || num_pages > INT32_MAX)
        return nullptr;
    for (int i = 0; i < n_caps; ++i)
        if (chunk_caps[i] < 1)
            return nullptr;
    cpsa_sched *h = new (std::nothrow) cpsa_sched();
    if (!h)
        return nullptr;
    h->budget = token_budget;
    h->page_size = page_size;
    h->caps.assign(chunk_caps, chunk_caps + n_caps);
    h->tile_align = tile_align;
    for (int64_t i = 0; i < num_pages; ++i)
        h->free_pages.push_back(page_order ? page_order[i] : (int32_t)i);
    return h;
}

void cpp_sched_destroy(cpsa_sched *h) { delete h; }

int cpp_sched_add_request(cpsa_sched *h, int64_t id, int64_t prompt_len, int64_t max_new_tokens)
{
    if (!h || prompt_len < 1 || max_new_tokens < 0)
        return CPSA_ERR_BAD_SHAPE;
    Request r;
    r.id = id;
    r.prompt_len = prompt_len;
    r.max_new = max_new_tokens;
    h->waiting.push_back(r);
    return CPSA_OK;
}

int cpp_sched_step(cpsa_sched *h, int max_reqs, int64_t max_tokens, int max_blocks, int64_t *req_ids,
                   int32_t *query_lens, int32_t *seq_lens, int32_t *block_table, int64_t *slot_mapping,
                   int *n_reqs, int64_t *n_tokens)
{
    if (!h || !n_reqs || !n_tokens || max_reqs < 0 || max_tokens < 0 || max_blocks < 1)
        return CPSA_ERR_BAD_SHAPE;
    if (h->pending)
        return CPSA_ERR_BAD_SHAPE;   // the previous step was not committed
    std::vector<Entry> batch;
    int64_t budget = h->budget;
    int64_t free_pages = (int64_t)h->free_pages.size();
    auto take = [&](int idx, int64_t tokens, bool decode) -> bool {
        const int64_t need = pages_needed(h, h->running[idx], tokens);
        if (need > free_pages)
            return false;
        free_pages -= need;
        batch.push_back(Entry{idx, tokens, decode});
        budget -= tokens;
        return true;
    };
    // 1. decode rows, one token each
    for (int i = 0; i < (int)h->running.size() && budget > 0; ++i) {
        const Request &r = h->running[i];
        if (r.prefilled == r.prompt_len && r.decoded < r.max_new)
            take(i, 1, true);
    }
    // 2. prompts already started
    for (int i = 0; i < (int)h->running.size() && budget > 0; ++i) {
        const Request &r = h->running[i];
        if (r.prefilled > 0 && r.prefilled < r.prompt_len) {
            const int64_t c = prefill_chunk(h, r, budget);
            if (c > 0)
                take(i, c, false);
        }
    }
    // 3. new requests in arrival order (admitted only if their first chunk fits);
    //    entry index running.size() + j stands for waiting[j] until the batch is applied
    const int base_idx = (int)h->running.size();
    int n_admit = 0;
    while (budget > 0 && n_admit < (int)h->waiting.size()) {
        const Request &r = h->waiting[n_admit];
        const int64_t c = prefill_chunk(h, r, budget);
        const int64_t need = c > 0 ? pages_needed(h, r, c) : 0;
        if (c <= 0 || need > free_pages)
            break;
        free_pages -= need;
        batch.push_back(Entry{base_idx + n_admit, c, false});
        budget -= c;
        ++n_admit;
    }
    auto req = [&](int idx) -> const Request & {
        return idx < base_idx ? h->running[idx] : h->waiting[idx - base_idx];
    };
    // check the caller's capacities before anything changes
    int64_t T = 0;
    for (const Entry &e : batch)
        T += e.tokens;
    if ((int)batch.size() > max_reqs || T > max_tokens)
        return CPSA_ERR_BAD_SHAPE;
    if ((!batch.empty()) && (!req_ids || !query_lens || !seq_lens || !block_table || (T > 0 && !slot_mapping)))
        return CPSA_ERR_NULL_ARG;
    for (const Entry &e : batch) {
        const int64_t s = req(e.idx).seq() + e.tokens;
        if ((s + h->page_size - 1) / h->page_size > max_blocks)
            return CPSA_ERR_BAD_SHAPE;
    }
    // apply: admit, allocate pages, write the step's metadata
    for (int j = 0; j < n_admit; ++j) {
        h->running.push_back(std::move(h->waiting.front()));
        h->waiting.pop_front();
    }
    int64_t t = 0;
    for (size_t b = 0; b < batch.size(); ++b) {
        const Entry &e = batch[b];
        Request &r = h->running[e.idx];
        const int64_t need = pages_needed(h, r, e.tokens);
        for (int64_t k = 0; k < need; ++k) {
            r.pages.push_back(h->free_pages.front());
            h->free_pages.pop_front();
        }
        const int64_t s0 = r.seq();
        req_ids[b] = r.id;
        query_lens[b] = (int32_t)e.tokens;
        seq_lens[b] = (int32_t)(s0 + e.tokens);
        int32_t *row = block_table + (int64_t)b * max_blocks;
        for (int k = 0; k < max_blocks; ++k)
            row[k] = k < (int)r.pages.size() ? r.pages[k] : -1;
        for (int64_t p = s0; p < s0 + e.tokens; ++p)
            slot_mapping[t++] = (int64_t)r.pages[p / h->page_size] * h->page_size + p % h->page_size;
    }
    h->last = batch;
    h->pending = true;
    *n_reqs = (int)batch.size();
    *n_tokens = T;
    return CPSA_OK;
}

int cpp_sched_commit(cpsa_sched *h)
{
    if (!h || !h->pending)
        return CPSA_ERR_BAD_SHAPE;
    for (const Entry &e : h->last) {
        Request &r = h->running[e.idx];
        if (e.decode) {
            r.decoded += 1;
        } else {
            r.prefilled += e.tokens;
            r.chunks += 1;
        }
    }
    // finished requests give their pages back (in order) and leave
    std::vector<Request> keep;
    keep.reserve(h->running.size());
    for (Request &r : h->running) {
        if (r.prefilled == r.prompt_len && r.decoded == r.max_new) {
            for (int32_t pg : r.pages)
                h->free_pages.push_back(pg);
            ++h->finished;
        } else {
            keep.push_back(std::move(r));
        }
    }
    h->running.swap(keep);
    h->last.clear();
    h->pending = false;
    return CPSA_OK;
}

int cpp_sched_stats(const cpsa_sched *h, int64_t *waiting, int64_t *running, int64_t *finished, int64_t *free_pages)
{
    if (!h)
        return CPSA_ERR_NULL_ARG;
    if (waiting)
        *waiting = (int64_t)h->waiting.size();
    if (running)
        *running = (int64_t)h->running.size();
    if (finished)
        *finished = h->finished;
    if (free_pages)
        *free_pages = (int64_t)h->free_pages.size();
    return CPSA_OK;
}

}  // extern "C"
