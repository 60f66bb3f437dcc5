"""Host-side checks of the seeded workloads and the harness page allocator (CPU only)."""
import numpy as np
import pytest

from conftest import golden_lines
from oracle.plan import computed_tokens, sharing_plan
from workloads import BF16_NAN, OutOfPages, PageAllocator, config_case


def test_allocator_grows_by_whole_pages_and_raises_when_exhausted():
    # "KV Cache Management and PagedAttention", "Grow the allocation as generation
    # proceeds": with 4-slot blocks, going from 7 to 8 positions needs no new block; the
    # 9th position takes a new one.
    a = PageAllocator(6, 4, permutation=[3, 0, 5, 1, 4, 2])
    a.reserve(0, 7)
    assert a.pages[0] == [3, 0]
    a.reserve(0, 1)
    assert a.pages[0] == [3, 0]
    a.reserve(0, 1)
    assert a.pages[0] == [3, 0, 5]
    a.reserve(1, 12)
    with pytest.raises(OutOfPages):
        a.reserve(2, 1)


def test_truncate_returns_pages_and_copies_nothing():
    a = PageAllocator(64, 16, permutation=np.arange(64))
    a.reserve(0, 350)
    assert len(a.pages[0]) == 22
    kept = list(a.pages[0][:19])
    a.truncate(0, 300)
    assert a.pages[0] == kept and len(a.free) == 64 - 19
    b = PageAllocator(16, 64, permutation=np.arange(16))
    b.reserve(0, 350)
    b.truncate(0, 300)
    assert len(b.pages[0]) == 5
    b.release(0)
    assert len(b.free) == 16


def test_shared_pages_are_freed_by_the_last_holder():
    a = PageAllocator(8, 4, permutation=np.arange(8))
    a.reserve(0, 8)
    a.share(1, 0, 8)
    a.reserve(1, 1)
    assert a.pages[1][:2] == a.pages[0]
    a.release(0)
    assert sorted(a.free) == [3, 4, 5, 6, 7]
    a.release(1)
    assert len(a.free) == 8


def test_config1_shape_and_poison():
    c = config_case(1)
    assert c.context_lens.tolist() == [1, 17, 33, 100]
    assert c.num_pages == 32 and c.block_table.shape == (4, 32)
    assert c.q.shape == (4, 4, 64) and c.k_new.shape == (4, 2, 64)
    pages = c.block_table
    # all 13 held pages are distinct, drawn from a permutation of the 32
    held = np.concatenate([pages[s, : -(-int(n) // 16)] for s, n in enumerate(c.context_lens)])
    assert len(set(held.tolist())) == 13
    # unheld pages are poison everywhere
    unheld = np.setdiff1d(np.arange(32), held)
    assert (c.k_pool[unheld] == BF16_NAN).all() and (c.v_pool[unheld] == BF16_NAN).all()
    # sequence 0 (ctx 1) has no cached position: its page is all poison until the store
    assert (c.k_pool[pages[0, 0]] == BF16_NAN).all()


def test_config_generation_is_deterministic():
    a, b = config_case(1), config_case(1)
    for f in ("q", "k_pool", "v_pool", "k_new", "v_new", "block_table"):
        assert np.array_equal(getattr(a, f), getattr(b, f))


def test_rewind_config_token_counts():
    g = {ln.split()[0]: int(ln.split()[1]) for ln in golden_lines("rewind_counts.txt")}
    c = config_case(4, num_seqs=g["documents"] // 10)
    assert c.num_tokens * 10 == g["new_tokens_with_rewind"]
    assert int(c.context_lens.sum()) * 10 == g["new_tokens_without_rewind"]
    assert (c.context_lens - c.q_lens == g["document_tokens"]).all()
    assert (c.q_lens == g["question_tokens"]).all()


def test_shared_prefix_config_matches_the_sharing_plan():
    c = config_case(3, num_seqs=32)
    order, parent, shared = sharing_plan(c.docs, c.page_size)
    for group in c.groups:
        leader = group[0]
        assert shared[leader] == 0 and parent[leader] is None
        for m in group[1:]:
            assert shared[m] == 2048 and parent[m] == leader
            assert np.array_equal(c.block_table[m, :128], c.block_table[leader, :128])
            assert not set(c.block_table[m, 128: -(-int(c.context_lens[m]) // 16)]) & set(
                c.block_table[leader, : -(-int(c.context_lens[leader]) // 16)])
    assert computed_tokens(c.docs, shared) == int(c.context_lens.sum()) - 2048 * 7 * 4


def test_copy_on_write_follows_the_worked_example():
    """PageAllocator.fork / reserve against the copy-on-write example of "KV Cache Management
    and PagedAttention" ("Split shared blocks when a write is needed", Figure 6)."""
    from conftest import golden_lines

    rows = [ln.split(" | ") for ln in golden_lines("copy_on_write.txt")]
    for common, prefix in ((6, ""), (8, "full-")):
        a = PageAllocator(8, 4, permutation=np.arange(8))
        a.reserve(0, common)                      # the common input: P0, P1
        a.fork(1, 0)                              # response 2 shares both blocks
        p0, p1 = a.pages[0]
        named = {p0: "P0", p1: "P1"}
        steps = [r for r in rows if r[0].startswith(prefix) and
                 (prefix or not r[0].startswith("full-"))]
        for step, writer, copies, physical, rc0, rc1 in steps:
            made = []
            if writer != "-":
                seq = int(writer) - 1
                for src, dst in a.reserve(seq, 1):
                    named.setdefault(dst, f"P{len(named)}")
                    made.append(f"{named[src]}->{named[dst]}")
            assert (",".join(made) or "-") == copies, step
            assert a.physical_pages() == int(physical), step
            assert a.refcount[p0] == int(rc0) and a.refcount[p1] == int(rc1), step
        # P0 is still in both tables; each response ends with its own last block
        assert a.pages[0][0] == a.pages[1][0] == p0
        assert a.pages[0][-1] != a.pages[1][-1]


def test_copy_on_write_oracle_copies_whole_pages():
    """oracle.copy_pages: destinations receive the sources' bits (NaN payloads included),
    every other page keeps its bits, and all copies read the pools as before the call."""
    from oracle import oracle

    rng = np.random.default_rng(5)
    k = rng.integers(0, 1 << 16, size=(10, 4, 2, 8), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(10, 4, 2, 8), dtype=np.uint16)
    k[3, 1, 0, 0] = 0x7FC1                       # a NaN with a payload
    k0, v0 = k.copy(), v.copy()
    src, dst = np.array([3, 7, 2]), np.array([5, 2, 9])   # page 2 is read and written
    oracle.copy_pages(k, v, src, dst)
    for s_, d_ in zip(src, dst):
        assert np.array_equal(k[d_], k0[s_]) and np.array_equal(v[d_], v0[s_])
    for p in set(range(10)) - set(dst.tolist()):
        assert np.array_equal(k[p], k0[p]) and np.array_equal(v[p], v0[p])
