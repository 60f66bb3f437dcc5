"""Pins of the oracle's groups-from-block-tables (CPU).  Expected values are worked out by
hand from the definition (adjacent tables, shareable pages before the last position's page,
runs cut at max_members, singletons dropped, prefix = smallest agreement in the chunk), from
the construction of the shared-prefix workload, and from invariance under relabelling pages."""
import numpy as np
import pytest

from oracle.plan import groups_from_block_tables, shareable_pages
from workloads import config_case

# P = 16.  s0/s1 agree on pages 5, 6, 7 (both can share 3 pages: ctx 60 -> 59 // 16, ctx 64
# -> 63 // 16); s2 can share only 2 (ctx 40) and agrees on 5, 6; s3 starts a new run (page
# 1); s4 can share 1 page (ctx 17) and agrees on it; s5 can share none (ctx 1).
BT = [[5, 6, 7, 8], [5, 6, 7, 9], [5, 6, 2, 3], [1, 2, 3, 4], [1, 2, 8, 8], [9, 9, 9, 9]]
CTX = [60, 64, 40, 50, 17, 1]


def test_shareable_pages():
    assert [shareable_pages(c, 16, 4) for c in CTX] == [3, 3, 2, 3, 1, 0]
    assert shareable_pages(0, 16, 4) == 0
    assert shareable_pages(1000, 16, 4) == 4          # at most the table's width


def test_hand_example():
    assert groups_from_block_tables(BT, CTX, 16, 8) == ([0, 3, 5], [0, 1, 2, 3, 4], [32, 16])


def test_hand_example_cut_at_two_members():
    # run [0, 3) -> chunks [0, 1] (agree on 3 pages) and [2] (alone); run [3, 5) -> [3, 4]
    assert groups_from_block_tables(BT, CTX, 16, 2) == ([0, 2, 4], [0, 1, 3, 4], [48, 16])


def test_no_sharing_and_empty():
    assert groups_from_block_tables([[1, 2], [3, 4], [5, 6]], [30, 30, 30], 16, 8) == \
        ([0], [], [])
    assert groups_from_block_tables([], [], 16, 8) == ([0], [], [])
    # equal tables, but neither sequence has a page before its last position's page
    assert groups_from_block_tables([[1, 2], [1, 2]], [16, 16], 16, 8) == ([0], [], [])


def test_shared_prefix_workload_groups():
    """The shared-prefix workload builds 32 groups of 8 whose tables share 128 pages and then
    diverge, the groups on disjoint pages: the tables give back exactly those groups."""
    case = config_case(3)
    indptr, seqs, prefix = groups_from_block_tables(case.block_table, case.context_lens,
                                                    case.page_size, 16)
    assert len(prefix) == 32 and prefix == [2048] * 32
    assert indptr == list(range(0, 257, 8))
    assert [sorted(seqs[indptr[g]:indptr[g + 1]]) for g in range(32)] == \
        [sorted(int(m) for m in grp) for grp in case.groups]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_relabelling_pages_changes_nothing(seed):
    rng = np.random.default_rng(seed)
    S, W = 40, 12
    base = rng.integers(0, 6, size=(S, W))
    base[rng.random(S) < 0.5] = base[0]              # many rows agree with row 0
    ctx = rng.integers(0, W * 16 + 1, size=S)
    relabel = rng.permutation(64)
    a = groups_from_block_tables(base.tolist(), ctx.tolist(), 16, 5)
    b = groups_from_block_tables(relabel[base].tolist(), ctx.tolist(), 16, 5)
    assert a == b
