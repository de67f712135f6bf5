"""Token-budget batch builder with page allocation (TEST INFRASTRUCTURE).

Follows the "vLLM Chunked-Prefills" article, section 3 (non-blocking
scheduling: a token budget per cycle; decode requests first, one token each;
then the unfinished prefills, min(remaining, budget) each; then new requests
while budget is left) and section 3.2.2 (chunk-size strategies: a progressive
list of caps such as [2048, 1024, 512], tile alignment of the chunk size).

Readings where the page is silent:
  * the progressive strategy caps a prompt's i-th chunk by caps[min(i, n-1)]
    (the last size repeats);
  * tile alignment rounds a chunk that is not its prompt's last down to a
    multiple of the tile (the page's 512 vs 513 example is about a chunk's size);
  * pages: every request keeps the pages of its sequence in order; new tokens
    take pages from the front of a free list, finished requests (prompt done and
    max_new_tokens decode rows run) return theirs to the back; a decode row or a
    started prompt that does not fit is skipped for the cycle, admission stops at
    the first new request whose first chunk does not fit;
  * a decode row processes the token produced by the previous step at position
    seq (the prompt's last chunk produces the first one).

Pinned by the page's cycle on hand cases, by invariants (budget never exceeded,
every token of every prompt scheduled exactly once, slots consistent with the
block table, no page held twice) and by the progressive and alignment rules.
"""
from __future__ import annotations

from collections import deque


class Request:
    def __init__(self, rid, prompt_len, max_new):
        self.id, self.prompt_len, self.max_new = rid, prompt_len, max_new
        self.prefilled = 0
        self.decoded = 0
        self.chunks = 0
        self.pages = []

    @property
    def seq(self):
        return self.prefilled + self.decoded


class Scheduler:
    def __init__(self, token_budget, page_size, num_pages, page_order=None, chunk_caps=(), tile_align=0):
        self.budget = token_budget
        self.P = page_size
        self.caps = list(chunk_caps)
        self.tile = tile_align
        self.free = deque(list(page_order) if page_order is not None else range(num_pages))
        self.waiting = deque()
        self.running = []
        self.last = None
        self.finished = 0

    def add_request(self, rid, prompt_len, max_new):
        self.waiting.append(Request(rid, prompt_len, max_new))

    def _chunk(self, r, budget):
        rem = r.prompt_len - r.prefilled
        c = min(rem, budget)
        if self.caps:
            c = min(c, self.caps[min(r.chunks, len(self.caps) - 1)])
        if c < rem and self.tile > 0:
            c -= c % self.tile
        return max(c, 0)

    def _need(self, r, tokens):
        pages = -(-(r.seq + tokens) // self.P)
        return max(0, pages - len(r.pages))

    def step(self):
        """The cycle's batch: list of (request, tokens, is_decode), metadata applied."""
        budget = self.budget
        free = len(self.free)
        batch = []
        for r in self.running:                                  # decode rows
            if budget <= 0:
                break
            if r.prefilled == r.prompt_len and r.decoded < r.max_new:
                need = self._need(r, 1)
                if need <= free:
                    free -= need
                    batch.append((r, 1, True))
                    budget -= 1
        for r in self.running:                                  # prompts already started
            if budget <= 0:
                break
            if 0 < r.prefilled < r.prompt_len:
                c = self._chunk(r, budget)
                if c > 0:
                    need = self._need(r, c)
                    if need <= free:
                        free -= need
                        batch.append((r, c, False))
                        budget -= c
        while budget > 0 and self.waiting:                      # new requests
            r = self.waiting[0]
            c = self._chunk(r, budget)
            if c <= 0 or self._need(r, c) > free:
                break
            free -= self._need(r, c)
            self.waiting.popleft()
            self.running.append(r)
            batch.append((r, c, False))
            budget -= c
        # metadata: pages for the new tokens, then the arrays of the step
        out = {"req_ids": [], "query_lens": [], "seq_lens": [], "block_table": [], "slot_mapping": []}
        for r, c, _ in batch:
            for _ in range(self._need(r, c)):
                r.pages.append(self.free.popleft())
            s0 = r.seq
            out["req_ids"].append(r.id)
            out["query_lens"].append(c)
            out["seq_lens"].append(s0 + c)
            out["block_table"].append(list(r.pages))
            out["slot_mapping"] += [r.pages[p // self.P] * self.P + p % self.P for p in range(s0, s0 + c)]
        self.last = batch
        return out

    def commit(self):
        for r, c, dec in self.last:
            if dec:
                r.decoded += 1
            else:
                r.prefilled += c
                r.chunks += 1
        keep = []
        for r in self.running:
            if r.prefilled == r.prompt_len and r.decoded == r.max_new:
                self.free.extend(r.pages)
                self.finished += 1
            else:
                keep.append(r)
        self.running = keep
        self.last = None
