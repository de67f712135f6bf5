"""Micro-batch split points (TEST INFRASTRUCTURE; pure Python integers).

Follows the Ascend dual-stream article, section 3.1 "choosing the split point":

* simple method: batch split = batch_size // 2, token split = sum of the first
  batch-split query_lens;
* balanced method: aim at half the total tokens, walk the cumulative query_lens,
  take the request boundary whose cumulative count is nearest that aim, and give
  up on two streams when the two halves differ by more than balance_threshold
  (relative to the smaller half) or when either half is below length_threshold.

Readings where the page is silent:
  * candidate boundaries are k = 1 .. B-1 (each micro-batch keeps >= 1 request);
  * ties in the distance go to the smallest k;
  * "seq_len1 / seq_len2" in the balance test are the two halves' token counts;
  * a half with zero tokens counts as unbalanced; B < 2 gives (0, 0, False).

Pinned by: hand cases, brute force over every k, and the 2600-prompt workload
(k* = 160, n1 = 83328) in tests/test_oracle_split_planner.py.
"""
from __future__ import annotations


def simple_split(query_lens):
    """(batch_split, token_split) by the simple method."""
    b = len(query_lens) // 2
    return b, int(sum(int(x) for x in query_lens[:b]))


def balanced_split(query_lens, balance_threshold: float, length_threshold: int):
    """(batch_split, token_split, use_two) by the balanced method."""
    q = [int(x) for x in query_lens]
    B = len(q)
    if B < 2:
        return 0, 0, False
    total = sum(q)
    best = total // 2
    cum = 0
    best_k = -1
    best_diff = None
    for k in range(1, B):
        cum += q[k - 1]
        diff = abs(cum - best)
        if best_diff is None or diff < best_diff:
            best_diff = diff
            best_k = k
    n1 = sum(q[:best_k])
    n2 = total - n1
    small = min(n1, n2)
    if small <= 0:
        return best_k, n1, False
    balanced = abs(n1 - n2) / small <= balance_threshold
    long_enough = small >= length_threshold
    return best_k, n1, bool(balanced and long_enough)
