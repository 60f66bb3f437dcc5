"""Quail's prefix-sharing plan, written out step by step (pure Python).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: Quail "KV", section "The sharing plan": documents are sorted by token sequence,
adjacent documents are compared for a common prefix, only complete pages are shared, the
final token of every document is left to be computed, and when the preceding document's
own shared count already covers the current one, the plan follows parent links back to the
document that supplies those pages.

Readings where the section leaves a step open:
  * sorting is a stable lexicographic sort of the token sequences;
  * the final-token cap comes before rounding down to whole pages:
    shared = floor(min(lcp, len - 1) / page_size) * page_size;
  * the preceding document covers the current one when its own shared count is at least
    the current one's; links are followed while that holds;
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


# --------------------------------------------------------------------------------------------
# Groups of sequences from their block tables (the grouped decode's device prepass).
#
# The sharing plan above decides which pages a document may take from another; once the
# tables exist, the sequences that do share pages can be found again from the tables alone.
# Readings (the pages give the plan, not this inverse):
#   * a sequence can share only whole pages that lie before the page holding its last
#     position (its newest token is stored into a page of its own; the plan likewise leaves
#     the final token to be computed): shareable(ctx) = floor((ctx - 1) / page_size), 0 for an
#     empty sequence, at most the table's width;
#   * adjacent sequences s - 1, s are linked when their tables agree on at least the first
#     shareable page; lcp(s) is the number of leading shareable pages on which they agree;
#   * a group is a maximal run of linked sequences, cut into consecutive chunks of at most
#     `max_members` (the grouped decode's row limit); a chunk of one sequence is no group;
#   * a group's prefix is the pages all its members agree on: the smallest lcp inside the
#     chunk (agreement is transitive along the run), in positions (pages * page_size).
# --------------------------------------------------------------------------------------------
def shareable_pages(ctx: int, page_size: int, width: int) -> int:
    return min(max(int(ctx) - 1, 0) // page_size, width)


def groups_from_block_tables(block_table, context_lens, page_size: int, max_members: int):
    """Return (group_indptr, group_seqs, prefix_len) as lists of int."""
    S = len(context_lens)
    width = len(block_table[0]) if S else 0
    lcp = [0] * S
    for s in range(1, S):
        lim = min(shareable_pages(context_lens[s - 1], page_size, width),
                  shareable_pages(context_lens[s], page_size, width))
        k = 0
        while k < lim and int(block_table[s - 1][k]) == int(block_table[s][k]):
            k += 1
        lcp[s] = k
    indptr, seqs, prefix = [0], [], []
    s = 0
    while s < S:
        e = s + 1
        while e < S and lcp[e] >= 1:
            e += 1                                  # the run is [s, e)
        for c in range(s, e, max_members):
            members = list(range(c, min(c + max_members, e)))
            if len(members) >= 2:
                seqs.extend(members)
                indptr.append(len(seqs))
                prefix.append(page_size * min(lcp[m] for m in members[1:]))
        s = e
    return indptr, seqs, prefix
