"""Quail's prefix-sharing plan, written out step by step (pure Python).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: Quail "KV", section "The sharing plan": documents are sorted by token sequence,
adjacent documents are compared for a common prefix, only complete pages are shared, the
final token of every document is left to be computed, and when the preceding document
reuses the whole shared prefix itself the plan follows parent links to the document that
supplies those pages.

Readings where the section leaves a step open:
  * sorting is a stable lexicographic sort of the token sequences;
  * the final-token cap comes before rounding down to whole pages:
    shared = floor(min(lcp, len - 1) / page_size) * page_size;
  * the preceding document "reuses the entire shared prefix" when its own shared count is
    at least the current one; links are followed while that holds;
  * a document that shares nothing has parent None.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple


def common_prefix_length(a: Sequence[int], b: Sequence[int]) -> int:
    n = 0
    for x, y in zip(a, b):
        if x != y:
            break
        n += 1
    return n


def sharing_plan(docs: Sequence[Sequence[int]], page_size: int
                 ) -> Tuple[List[int], List[Optional[int]], List[int]]:
    """Return (order, parent, shared); parent and shared are indexed by document id."""
    order = sorted(range(len(docs)), key=lambda i: list(docs[i]))  # sorted() is stable
    parent: List[Optional[int]] = [None] * len(docs)
    shared = [0] * len(docs)
    for k in range(1, len(order)):
        doc, prev = order[k], order[k - 1]
        lcp = common_prefix_length(docs[doc], docs[prev])
        capped = min(lcp, len(docs[doc]) - 1)          # leave the final token to compute
        shared[doc] = (max(capped, 0) // page_size) * page_size   # complete pages only
        if shared[doc] == 0:
            continue
        p = prev
        while shared[p] >= shared[doc] and parent[p] is not None:
            p = parent[p]                               # follow the supplier of the pages
        parent[doc] = p
    return order, parent, shared


def computed_tokens(docs: Sequence[Sequence[int]], shared: Sequence[int]) -> int:
    """Document tokens that must still be processed when the plan's KV is available."""
    return sum(len(d) - s for d, s in zip(docs, shared))
