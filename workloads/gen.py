"""Seeded generators: bf16 draws, a host page allocator and test-case assembly.

Nothing here computes a slot, a score or an output.  The allocator knows, as any page
allocator does, which pages a sequence holds and how many of their positions are filled;
that is what decides which pool entries hold data and which hold the NaN poison.
"""
from __future__ import annotations

import concurrent.futures as futures
import os
from dataclasses import dataclass, field
from typing import Callable, Dict, List, Optional, Sequence, Tuple

import numpy as np

BF16_NAN = 0x7FC0          # quiet NaN in bf16; poisons every pool entry that holds no position
_CHUNK = 1 << 24            # elements per independently seeded draw chunk
_normal_table: Optional[np.ndarray] = None


def bf16_bits(x) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + (((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF))) >> np.uint32(16)
    return r.astype(np.uint16)


def f32_from_bf16(bits) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _table() -> np.ndarray:
    """bf16 patterns of the N(0,1) quantiles at (i + 1/2) / 65536, i = 0 .. 65535."""
    global _normal_table
    if _normal_table is None:
        from scipy.special import ndtri
        q = ndtri((np.arange(65536, dtype=np.float64) + 0.5) / 65536.0)
        _normal_table = bf16_bits(q.astype(np.float32))
    return _normal_table


def normal_bf16(seed: np.random.SeedSequence, shape) -> np.ndarray:
    """bf16 draws from N(0,1) by inverse-transform sampling of a 16-bit uniform code.

    Chunk c of _CHUNK elements is drawn from the c-th child of ``seed``, so the result does
    not depend on how many threads fill it.  Tails are cut at about 4.3 sigma.
    """
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    n_chunks = max(1, -(-n // _CHUNK))
    children = seed.spawn(n_chunks)
    table = _table()

    def fill(c: int) -> None:
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        codes = np.random.default_rng(children[c]).integers(0, 65536, size=hi - lo,
                                                            dtype=np.uint16)
        out[lo:hi] = table[codes]

    if n_chunks == 1:
        fill(0)
    else:
        workers = min(n_chunks, os.cpu_count() or 1, 16)
        with futures.ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out.reshape(shape)


class OutOfPages(RuntimeError):
    """The pool has no free page left (TileInfer.jl's OutOfPagesError)."""


class PageAllocator:
    """Host page allocator: a stack of free page ids, per-sequence page lists, refcounts.

    Mirrors TileInfer.jl "KV cache", section "Growing, rolling back, releasing":
    ``reserve`` gives a sequence pages for its next n positions and raises OutOfPages when
    the pool is exhausted; ``truncate`` keeps the first n positions and returns the pages
    no longer needed, copying and clearing nothing; ``release`` returns every page.
    Pages listed by several sequences (a shared prefix) are freed when the last holder
    lets go ("KV Cache Management and PagedAttention", section "Return blocks after a
    request ends").  The stack starts in the order of a seeded permutation, so tables point
    at scattered pages.
    """

    def __init__(self, num_pages: int, page_size: int, permutation: Sequence[int]):
        self.num_pages = int(num_pages)
        self.page_size = int(page_size)
        self.free: List[int] = [int(p) for p in reversed(list(permutation))]
        self.refcount = np.zeros(self.num_pages, dtype=np.int64)
        self.pages: Dict[int, List[int]] = {}
        self.length: Dict[int, int] = {}

    def _pop(self) -> int:
        if not self.free:
            raise OutOfPages(f"all {self.num_pages} pages are in use")
        page = self.free.pop()
        self.refcount[page] += 1
        return page

    def _drop(self, page: int) -> None:
        self.refcount[page] -= 1
        if self.refcount[page] == 0:
            self.free.append(page)

    def pages_for(self, positions: int) -> int:
        return -(-int(positions) // self.page_size)

    def reserve(self, seq: int, n: int) -> List[Tuple[int, int]]:
        """Room for the sequence's next n positions.  Returns the page copies (src, dst) the
        caller must make before writing: when the first new position falls inside a partly
        filled last page that other sequences still reference, that page is copied to a new
        one and the sequence's entry points at the copy ("KV Cache Management and
        PagedAttention", section "Split shared blocks when a write is needed"); a full shared
        page stays shared, and the new positions go to new pages."""
        pages = self.pages.setdefault(seq, [])
        length = self.length.get(seq, 0)
        need = self.pages_for(length + n) - len(pages)
        cow = n > 0 and length % self.page_size != 0 and self.refcount[pages[-1]] > 1
        if need + int(cow) > len(self.free):
            raise OutOfPages(f"sequence {seq} needs {need + int(cow)} pages, "
                             f"{len(self.free)} free")
        copies: List[Tuple[int, int]] = []
        if cow:
            old = pages[-1]
            pages[-1] = self._pop()
            self._drop(old)
            copies.append((old, pages[-1]))
        for _ in range(need):
            pages.append(self._pop())
        self.length[seq] = length + n
        return copies

    def fork(self, seq: int, donor: int) -> None:
        """Start ``seq`` on every page of the donor, a partly filled last page included (two
        responses continuing one common input)."""
        assert seq not in self.pages
        for page in self.pages[donor]:
            self.refcount[page] += 1
        self.pages[seq] = list(self.pages[donor])
        self.length[seq] = self.length[donor]

    def physical_pages(self) -> int:
        """Pages referenced by at least one sequence."""
        return int(np.count_nonzero(self.refcount))

    def share(self, seq: int, donor: int, positions: int) -> None:
        """Start ``seq`` on the donor's first ``positions`` (a whole number of pages)."""
        assert positions % self.page_size == 0 and seq not in self.pages
        shared = self.pages[donor][: positions // self.page_size]
        for page in shared:
            self.refcount[page] += 1
        self.pages[seq] = list(shared)
        self.length[seq] = positions

    def truncate(self, seq: int, n: int) -> None:
        pages = self.pages[seq]
        keep = self.pages_for(n)
        for page in reversed(pages[keep:]):
            self._drop(page)
        del pages[keep:]
        self.length[seq] = min(self.length[seq], n)

    def release(self, seq: int) -> None:
        for page in reversed(self.pages.pop(seq, [])):
            self._drop(page)
        self.length.pop(seq, None)

    def table(self, seqs: Sequence[int], width: int) -> np.ndarray:
        """Fixed-width block table, zero padded (TileInfer.jl: padding entries are page 0)."""
        bt = np.zeros((len(seqs), width), dtype=np.int32)
        for row, seq in enumerate(seqs):
            pages = self.pages.get(seq, [])
            assert len(pages) <= width, "block table row too short"
            bt[row, : len(pages)] = pages
        return bt


@dataclass
class Case:
    """One batch of synthetic input.  bf16 tensors are held as uint16 bit patterns."""
    name: str
    page_size: int
    q_heads: int
    kv_heads: int
    head_dim: int
    num_pages: int
    context_lens: np.ndarray      # int32 [S], includes the new tokens
    q_indptr: np.ndarray          # int32 [S+1]
    block_table: np.ndarray       # int32 [S, W]
    q: np.ndarray                 # uint16 [T, Hq, D]
    k_new: np.ndarray             # uint16 [T, Hkv, D]
    v_new: np.ndarray             # uint16 [T, Hkv, D]
    k_pool: np.ndarray            # uint16 [num_pages, P, Hkv, D]
    v_pool: np.ndarray            # uint16 [num_pages, P, Hkv, D]
    allocator: Optional[PageAllocator] = None
    seqs: List[int] = field(default_factory=list)
    docs: Optional[List[np.ndarray]] = None      # token ids, where the case has them
    groups: Optional[List[List[int]]] = None     # sequences that share a prefix
    shared_positions: object = 0                 # per group (or one value for all groups)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q_indptr[-1])

    @property
    def max_ctx(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def max_q_len(self) -> int:
        return int(np.diff(self.q_indptr).max()) if self.num_seqs else 0

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.q_indptr).astype(np.int32)


def round_up(x: int, m: int) -> int:
    return -(-int(x) // m) * m


def _poison_unfilled(pool_k: np.ndarray, pool_v: np.ndarray, alloc: PageAllocator,
                     seqs: Sequence[int], filled: Sequence[int]) -> None:
    """NaN every pool entry that holds no filled position of any sequence."""
    P = alloc.page_size
    live = np.zeros((alloc.num_pages, P), dtype=bool)
    offsets = np.arange(P)
    for seq, n_filled in zip(seqs, filled):
        pages = np.asarray(alloc.pages.get(seq, []), dtype=np.int64)
        if pages.size == 0:
            continue
        per_page = np.clip(n_filled - np.arange(pages.size) * P, 0, P)
        live[pages] |= offsets[None, :] < per_page[:, None]
    pool_k[~live] = BF16_NAN
    pool_v[~live] = BF16_NAN


def build_case(seed: int, *, name: str, page_size: int, q_heads: int, kv_heads: int,
               head_dim: int, context_lens: Callable[[np.random.Generator], np.ndarray],
               q_lens: Callable[[np.ndarray], np.ndarray], num_pages: Optional[int] = None,
               slack: float = 0.10, bt_width: Optional[int] = None,
               share_groups: Optional[Callable[[np.random.Generator, np.ndarray], dict]] = None,
               poison: bool = True) -> Case:
    """Assemble one case.

    Streams: SeedSequence(seed) spawns, in this order, the streams for the context lengths,
    the page permutation, Q, the cached K, the cached V, the new K/V and the token ids.
    Every sequence's positions 0 .. ctx - q_len - 1 are cached (random K/V); positions
    ctx - q_len .. ctx - 1 are the new tokens (their K/V are in k_new / v_new and their
    pool entries start as poison, to be written by a store).
    """
    root = np.random.SeedSequence(seed)
    s_ctx, s_perm, s_q, s_k, s_v, s_new, s_tok = root.spawn(7)
    ctx = np.asarray(context_lens(np.random.default_rng(s_ctx)), dtype=np.int32)
    qlen = np.asarray(q_lens(ctx), dtype=np.int32)
    S = ctx.shape[0]
    P = page_size
    sharing = share_groups(np.random.default_rng(s_tok), ctx) if share_groups else None
    shared_pos = sharing["shared_positions"] if sharing else 0
    group_shared = []
    if sharing:
        sp = sharing["shared_positions"]
        group_shared = [int(sp[i]) if np.ndim(sp) else int(sp)
                        for i in range(len(sharing["groups"]))]
    if num_pages is None:
        need = sum(-(-int(c) // P) for c in ctx)
        if sharing:
            need -= sum((len(g) - 1) * (sh // P) for g, sh in zip(sharing["groups"],
                                                                   group_shared))
        num_pages = max(1, int(np.ceil(need * (1.0 + slack))))
    alloc = PageAllocator(num_pages, P, np.random.default_rng(s_perm).permutation(num_pages))
    seqs = list(range(S))
    grouped = set()
    if sharing:
        for group, sh in zip(sharing["groups"], group_shared):
            leader = group[0]
            alloc.reserve(leader, int(ctx[leader]))
            grouped.add(leader)
            for member in group[1:]:
                alloc.share(member, leader, sh)
                alloc.reserve(member, int(ctx[member]) - sh)
                grouped.add(member)
    for s in seqs:
        if s not in grouped:
            alloc.reserve(s, int(ctx[s]))
    if bt_width is None:
        bt_width = round_up(max(1, max(len(alloc.pages[s]) for s in seqs) if S else 1), 16)
    bt = alloc.table(seqs, bt_width)
    q_indptr = np.zeros(S + 1, dtype=np.int32)
    q_indptr[1:] = np.cumsum(qlen)
    T = int(q_indptr[-1])
    q = normal_bf16(s_q, (T, q_heads, head_dim))
    k_pool = normal_bf16(s_k, (num_pages, P, kv_heads, head_dim))
    v_pool = normal_bf16(s_v, (num_pages, P, kv_heads, head_dim))
    new = normal_bf16(s_new, (2, T, kv_heads, head_dim))
    if poison:
        _poison_unfilled(k_pool, v_pool, alloc, seqs, [int(c - l) for c, l in zip(ctx, qlen)])
    return Case(name=name, page_size=P, q_heads=q_heads, kv_heads=kv_heads,
                head_dim=head_dim, num_pages=num_pages, context_lens=ctx, q_indptr=q_indptr,
                block_table=bt, q=q, k_new=np.ascontiguousarray(new[0]),
                v_new=np.ascontiguousarray(new[1]), k_pool=k_pool, v_pool=v_pool,
                allocator=alloc, seqs=seqs,
                docs=sharing.get("docs") if sharing else None,
                groups=sharing["groups"] if sharing else None,
                shared_positions=shared_pos)


def repoison(case: Case, filled: Optional[Sequence[int]] = None) -> None:
    """Re-poison pool entries after the allocator changed (e.g. after a truncate)."""
    if filled is None:
        filled = [int(c - l) for c, l in zip(case.context_lens, case.q_lens)]
    _poison_unfilled(case.k_pool, case.v_pool, case.allocator, case.seqs, filled)
