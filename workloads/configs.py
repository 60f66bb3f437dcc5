"""The five workloads, as seeded synthetic inputs.

Each is shaped like a workload on the pages:
  1 tiny decode       -- a handful of sequences, every tail case of the address rule
  2 batched decode    -- 64 sequences of 512..4096 positions, Llama-3-8B-shaped heads
  3 shared prefix     -- 32 groups of 8 sequences whose tables share 128 pages (Quail
                         "KV", "Prefix sharing"; "KV Cache Management and PagedAttention",
                         "Share common KV across responses")
  4 KV-rewind append  -- 1,000 documents of 300 cached tokens, each appending a 50-token
                         question (Quail "KV", "KV rewind"), page size 16 or 64
  5 long decode       -- 8 sequences of 32k..128k positions (TileInfer.jl "KV cache",
                         "Sizing": decode at 32k positions)
Config k uses seed 20261202 + k.
"""
from __future__ import annotations

import numpy as np

from .gen import Case, build_case, round_up

SEED_BASE = 20261202

CONFIGS = {
    1: dict(name="tiny-decode", page_size=16, q_heads=4, kv_heads=2, head_dim=64),
    2: dict(name="batched-decode", page_size=16, q_heads=32, kv_heads=8, head_dim=128),
    3: dict(name="shared-prefix-decode", page_size=16, q_heads=32, kv_heads=8,
            head_dim=128),
    4: dict(name="rewind-append", page_size=16, q_heads=32, kv_heads=8, head_dim=128),
    5: dict(name="long-decode", page_size=64, q_heads=64, kv_heads=8, head_dim=128),
}


def _decode_qlens(ctx):
    return np.ones_like(ctx)


def _shared_prefix_groups(n_groups: int, members: int, prefix: int, vocab: int = 32000):
    def make(rng: np.random.Generator, ctx: np.ndarray) -> dict:
        docs, groups = [], []
        for g in range(n_groups):
            head = rng.integers(n_groups, vocab, size=prefix)
            head[0] = g                     # distinct first token: groups share nothing
            group = []
            for m in range(members):
                s = g * members + m
                tail = rng.integers(members, vocab, size=int(ctx[s]) - prefix)
                tail[0] = m                 # distinct first suffix token inside the group
                docs.append(np.concatenate([head, tail]).astype(np.int64))
                group.append(s)
            groups.append(group)
        return dict(docs=docs, groups=groups, shared_positions=prefix)
    return make


def config_case(k: int, *, page_size: int = None, num_seqs: int = None,
                poison: bool = True, seed: int = None) -> Case:
    """Build config k.  ``page_size`` overrides config 4's page size (16 or 64);
    ``num_seqs`` shrinks configs 2-5 to fewer sequences / groups / documents (for quick
    checks; the full configs leave it None); ``seed`` replaces the config's seed (another
    batch drawn by the same recipe)."""
    cfg = dict(CONFIGS[k])
    name = cfg.pop("name")
    seed = SEED_BASE + k if seed is None else seed
    if k == 1:
        return build_case(seed, name=name, **cfg, num_pages=32, bt_width=32,
                          context_lens=lambda rng: np.array([1, 17, 33, 100]),
                          q_lens=_decode_qlens, poison=poison)
    if k == 2:
        S = num_seqs or 64
        return build_case(seed, name=name, **cfg, bt_width=256,
                          context_lens=lambda rng: rng.integers(512, 4097, size=S),
                          q_lens=_decode_qlens, poison=poison)
    if k == 3:
        n_groups = (num_seqs or 256) // 8
        S = n_groups * 8
        return build_case(seed, name=name, **cfg, bt_width=160,
                          context_lens=lambda rng: 2048 + rng.integers(64, 513, size=S),
                          q_lens=_decode_qlens,
                          share_groups=_shared_prefix_groups(n_groups, 8, 2048),
                          poison=poison)
    if k == 4:
        P = page_size or 16
        cfg["page_size"] = P
        S = num_seqs or 1000
        return build_case(seed, name=f"{name}-p{P}", **cfg,
                          bt_width=round_up(-(-350 // P), 16),
                          context_lens=lambda rng: np.full(S, 350),
                          q_lens=lambda ctx: np.full_like(ctx, 50), poison=poison)
    if k == 5:
        S = num_seqs or 8
        return build_case(seed, name=name, **cfg, bt_width=2048,
                          context_lens=lambda rng: rng.integers(32768, 131073, size=S),
                          q_lens=_decode_qlens, poison=poison)
    raise KeyError(k)
