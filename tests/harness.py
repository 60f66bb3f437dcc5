"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI, run the
oracle on the same seeded inputs, compare."""
from __future__ import annotations

import os

import numpy as np
import torch

import pagedattention_kvc_store_gb300 as kvc
from oracle import oracle
from workloads.device import bf16_bits_of, to_device

# Attention tolerance against the fp64 oracle (bf16 inputs, fp32 accumulation).
MAX_ABS = 1e-2
MEAN_ABS = 1e-3
THREADS = max(1, min(16, os.cpu_count() or 1))


def out_to_f64(out: torch.Tensor) -> np.ndarray:
    return out.float().cpu().numpy().astype(np.float64)


def assert_attention_close(got: np.ndarray, ref: np.ndarray, what: str = "",
                           max_abs: float = MAX_ABS, mean_abs: float = MEAN_ABS):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= max_abs, f"{what}: max abs error {err.max():.3e} > {max_abs}"
    assert err.mean() <= mean_abs, f"{what}: mean abs error {err.mean():.3e} > {mean_abs}"
    return float(err.max()), float(err.mean())


class GpuRun:
    """The CUDA path on one case: slot mapping -> store -> decode or append."""

    def __init__(self, case, decode: bool):
        self.case = case
        self.decode = decode
        self.d = to_device(case)
        self.slots = torch.empty(case.num_tokens, dtype=torch.int32, device="cuda")

    def store(self):
        c, d = self.case, self.d
        kvc.kvc_slot_mapping(self.slots, d.block_table, d.context_lens,
                             None if self.decode else d.q_indptr, c.page_size,
                             max_q_len=c.max_q_len)
        kvc.kvc_store(d.k_pool, d.v_pool, d.k_new, d.v_new, self.slots)

    def attend(self, out_dtype=torch.bfloat16, num_splits=0):
        c, d = self.case, self.d
        out = torch.empty((c.num_tokens, c.q_heads, c.head_dim), dtype=out_dtype,
                          device="cuda")
        if self.decode:
            pool = kvc.pool_desc(d.k_pool)
            _, _, ws = kvc.kvc_decode_plan(c.num_seqs, c.q_heads, pool, c.max_ctx, num_splits)
            self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
            kvc.kvc_decode(out, d.q, d.k_pool, d.v_pool, d.block_table, d.context_lens,
                           c.max_ctx, num_splits=num_splits, workspace=self.workspace)
        else:
            kvc.kvc_append(out, d.q, d.k_pool, d.v_pool, d.block_table, d.q_indptr,
                           d.context_lens, c.max_q_len, c.max_ctx)
        return out


class OracleRun:
    """The oracle on the same case: its own slot mapping, store and attention."""

    def __init__(self, case):
        self.case = case
        self.slots = oracle.slot_mapping(case.block_table, case.context_lens, case.q_indptr,
                                         case.page_size)
        self.k_pool = case.k_pool.copy()
        self.v_pool = case.v_pool.copy()
        oracle.store(self.k_pool, self.v_pool, case.k_new, case.v_new, self.slots)

    def attention(self, seqs=None):
        """(out, lse) for all sequences, or for the listed ones (rows of those only)."""
        c = self.case
        if seqs is None:
            return oracle.attention(c.q, self.k_pool, self.v_pool, c.block_table,
                                    c.context_lens, c.q_indptr, num_threads=THREADS)
        seqs = np.asarray(seqs)
        q_rows = np.concatenate([np.arange(c.q_indptr[s], c.q_indptr[s + 1]) for s in seqs])
        q_lens = (c.q_indptr[seqs + 1] - c.q_indptr[seqs]).astype(np.int32)
        indptr = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
        out, lse = oracle.attention(c.q[q_rows], self.k_pool, self.v_pool,
                                    c.block_table[seqs], c.context_lens[seqs], indptr,
                                    num_threads=THREADS)
        return out, lse, q_rows


def sample_seqs(n_total: int, n: int, seed: int = 0):
    if n >= n_total:
        return np.arange(n_total)
    return np.sort(np.random.default_rng(seed).choice(n_total, size=n, replace=False))


def pools_bits(run: GpuRun):
    return bf16_bits_of(run.d.k_pool), bf16_bits_of(run.d.v_pool)


def int8_pages(case, seed=0):
    """INT8 pools holding the case's cached positions (every live position except the new
    tokens'), poisoned elsewhere: random codes, NaN scales."""
    rng = np.random.default_rng(seed)
    pages, P, H, D = case.k_pool.shape
    kc = rng.integers(-128, 128, size=(pages, P, H, D)).astype(np.int8)
    vc = rng.integers(-128, 128, size=(pages, P, H, D)).astype(np.int8)
    ks = np.full((pages, H, P), np.nan, np.float32)
    vs = np.full((pages, H, P), np.nan, np.float32)
    slots = []
    for s in range(case.num_seqs):
        q_len = case.q_indptr[s + 1] - case.q_indptr[s]
        for p in range(case.context_lens[s] - q_len):
            slots.append(oracle.slot_of_position(case.block_table, s, p, P))
    slots = np.array(slots, dtype=np.int64)
    flat_k = case.k_pool.reshape(pages * P, H, D)
    flat_v = case.v_pool.reshape(pages * P, H, D)
    oracle.store_int8(kc, vc, ks, vs, flat_k[slots], flat_v[slots], slots)
    return kc, vc, ks, vs
