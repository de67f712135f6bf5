"""The token-budget batch builder: the oracle's cycle on hand cases and invariants,
and the library's (host C++) builder against the oracle on random request streams
(CPU only)."""
import numpy as np
import pytest

import oracle


def run_steps(sched, n):
    out = []
    for _ in range(n):
        out.append(sched.step())
        sched.commit()
    return out


def test_cycle_hand_case():
    """Budget 512: decode rows first, then the started prompt, then new requests."""
    s = oracle.Scheduler(512, 16, 256)
    s.add_request("A", 300, 3)
    s.add_request("B", 1000, 0)
    s.add_request("C", 100, 1)
    b1, b2, b3 = run_steps(s, 3)
    assert (b1["req_ids"], b1["query_lens"], b1["seq_lens"]) == (["A", "B"], [300, 212], [300, 212])
    # A is a decode row now (one token), B continues with the rest of the budget, C waits
    assert (b2["req_ids"], b2["query_lens"], b2["seq_lens"]) == (["A", "B"], [1, 511], [301, 723])
    # B has 277 left: A decodes, B finishes its prompt, C starts with the remaining 234
    assert (b3["req_ids"], b3["query_lens"], b3["seq_lens"]) == (["A", "B", "C"], [1, 277, 100], [302, 1000, 100])
    assert s.finished == 1        # B: prompt done, no decode rows asked
    for b in (b1, b2, b3):
        check_invariants(b, 512, 16, None)
    # pages: A holds ceil(302 / 16) = 19, C ceil(100 / 16) = 7; B's 63 came back
    assert len(s.free) == 256 - 19 - 7
    # the pages of a step's first request start the free list, in order
    assert b1["block_table"][0] == list(range(19)) and b1["slot_mapping"][:3] == [0, 1, 2]


def test_progressive_caps_and_tile_alignment():
    s = oracle.Scheduler(4096, 128, 1000, chunk_caps=[2048, 1024, 512])
    s.add_request(0, 8000, 0)
    sizes = []
    for _ in range(64):                     # 8000 tokens take 14 steps; bounded all the same
        if not (s.waiting or s.running):
            break
        sizes += s.step()["query_lens"]
        s.commit()
    assert not (s.waiting or s.running)
    assert sizes[:3] == [2048, 1024, 512] and set(sizes[3:-1]) == {512} and sum(sizes) == 8000
    # tile alignment: three decode rows leave 2045 tokens, rounded down to 1920
    s = oracle.Scheduler(2048, 16, 4096, tile_align=128)
    for i in range(3):
        s.add_request(i, 16, 5)
    s.add_request(9, 5000, 0)
    s.step(); s.commit()          # the three 16-token prompts and 2000 of the long one (not last: 1920)
    b = s.step()
    assert b["query_lens"][:3] == [1, 1, 1] and b["query_lens"][3] == 1920
    s.commit()
    # its last chunk is whatever remains, 5000 - 2 x 1920 = 1160, not rounded to the tile
    b = s.step()
    assert b["req_ids"][3] == 9 and b["query_lens"][3] == 1160


def check_invariants(batch, budget, P, live_pages):
    assert sum(batch["query_lens"]) <= budget
    t = 0
    for q, sl, bt in zip(batch["query_lens"], batch["seq_lens"], batch["block_table"]):
        for p in range(sl - q, sl):
            assert batch["slot_mapping"][t] == bt[p // P] * P + p % P
            t += 1
        assert len(bt) == -(-sl // P)
    pages = [pg for bt in batch["block_table"] for pg in bt]
    assert len(pages) == len(set(pages))


def random_stream(rng, n):
    return [(i, int(rng.integers(1, 3000)), int(rng.integers(0, 40))) for i in range(n)]


@pytest.mark.parametrize("budget,P,caps,tile,pages", [(512, 16, (), 0, 2048), (2048, 16, (2048, 1024, 512), 128, 900),
                                                      (2048, 128, (), 128, 300), (300, 8, (256, 64), 0, 3000)])
def test_library_builder_matches_oracle(budget, P, caps, tile, pages):
    import chunked_prefill_paged_slot_gb300 as cpsa
    rng = np.random.default_rng(budget + P + pages)
    order = rng.permutation(pages).astype(np.int32)
    ours = cpsa.BatchScheduler(budget, P, pages, page_order=order, chunk_caps=caps, tile_align=tile,
                               max_reqs=512, max_blocks=512)
    ref = oracle.Scheduler(budget, P, pages, page_order=order.tolist(), chunk_caps=caps, tile_align=tile)
    stream = random_stream(rng, 40)
    for rid, L, m in stream:
        ours.add_request(rid, L, m)
        ref.add_request(rid, L, m)
    steps, scheduled = 0, {}
    while ref.waiting or ref.running:
        a, b = ours.step(), ref.step()
        assert a["req_ids"].tolist() == b["req_ids"]
        assert a["query_lens"].tolist() == b["query_lens"]
        assert a["seq_lens"].tolist() == b["seq_lens"]
        assert a["slot_mapping"].tolist() == b["slot_mapping"]
        for r, row in enumerate(b["block_table"]):
            assert a["block_table"][r, :len(row)].tolist() == row
            assert (a["block_table"][r, len(row):] == -1).all()
        check_invariants(b, budget, P, None)
        for rid, q, sl in zip(b["req_ids"], b["query_lens"], b["seq_lens"]):
            scheduled[rid] = scheduled.get(rid, 0) + q
        ours.commit()
        ref.commit()
        steps += 1
        assert len(b["req_ids"]) > 0, "no progress"
    # every prompt token and decode row ran exactly once
    for rid, L, m in stream:
        assert scheduled[rid] == L + m
    assert ours.stats() == (0, 0, len(stream), pages)
    ours.close()


def test_library_builder_leaves_state_on_capacity_error():
    import chunked_prefill_paged_slot_gb300 as cpsa
    s = cpsa.BatchScheduler(512, 16, 128, max_reqs=1, max_blocks=64)
    s.add_request(1, 100, 0)
    s.add_request(2, 100, 0)
    with pytest.raises(cpsa.CpsaError):
        s.step()                      # two requests in the batch, room for one
    assert s.stats() == (2, 0, 0, 128)
    s.close()
