"""INT8 append on the GPU against the oracle (TileInfer.jl "KV cache", "INT8 cache"; causal
prefill as in Quail "KV", "KV rewind").

The cached positions of a seeded case are quantised into INT8 pages by the oracle; slots that
hold no position keep random codes and NaN scales.  The new tokens are quantised and stored by
kvc_store_int8 (codes and scales bit-exact against the oracle's store), then kvc_append_int8
attends causally over the pages; the oracle's fp64 attention over scale * code is the
reference, within the attention tolerance."""
import numpy as np
import pytest
import torch

import pagedattention_kvc_store_gb300 as kvc
from harness import (MAX_ABS, MEAN_ABS, assert_attention_close, int8_pages, out_to_f64,
                     sample_seqs)
from oracle import oracle
from workloads import build_case, config_case
from workloads.device import bf16_tensor, i32_tensor

pytestmark = pytest.mark.gpu


def assert_close_out(got, ref, what, dtype):
    """The attention tolerance; a bf16 output may in addition be off by its own rounding, half
    an ulp (at most 2^-8 |x|): unlike a bf16 cache, scale * code is seldom a bf16 number, so a
    context of one position already shows it."""
    if dtype == torch.float32:
        assert_attention_close(got, ref, what)
        return
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    excess = err - 2.0 ** -8 * np.abs(ref)
    assert excess.max() <= MAX_ABS, f"{what}: max error beyond rounding {excess.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean abs error {err.mean():.3e}"


class Int8AppendRun:
    """One case on the GPU: INT8 pools with the cached positions, the new tokens stored by
    kvc_store_int8 (checked against the oracle's store), ready for kvc_append_int8."""

    def __init__(self, case):
        self.case = case
        kc, vc, ks, vs = int8_pages(case)
        self.dev = [torch.from_numpy(a).cuda() for a in (kc, vc, ks, vs)]
        self.bt = i32_tensor(case.block_table, "cuda")
        self.ctx = i32_tensor(case.context_lens, "cuda")
        self.ind = i32_tensor(case.q_indptr, "cuda")
        slots = torch.empty(case.num_tokens, dtype=torch.int32, device="cuda")
        kvc.kvc_slot_mapping(slots, self.bt, self.ctx, self.ind, case.page_size,
                             max_q_len=case.max_q_len)
        kvc.kvc_store_int8(*self.dev, bf16_tensor(case.k_new, "cuda"),
                           bf16_tensor(case.v_new, "cuda"), slots)
        oracle.store_int8(kc, vc, ks, vs, case.k_new, case.v_new,
                          slots.cpu().numpy().astype(np.int64))
        for name, got, ref in zip(("K codes", "V codes", "K scales", "V scales"), self.dev,
                                  (kc, vc, ks, vs)):
            g = got.cpu().numpy()
            assert np.array_equal(g, ref, equal_nan=ref.dtype == np.float32), \
                f"{name} differ from the oracle's store"
        self.pools = (kc, vc, ks, vs)
        self.q = bf16_tensor(case.q, "cuda")

    def attend(self, dtype=torch.float32, scale=0.0):
        c = self.case
        out = torch.empty(c.num_tokens, c.q_heads, c.head_dim, dtype=dtype, device="cuda")
        kvc.kvc_append_int8(out, self.q, *self.dev, self.bt, self.ind, self.ctx, c.max_q_len,
                            c.max_ctx, scale=scale)
        torch.cuda.synchronize()
        assert kvc.kvc_device_errors() == 0
        return out_to_f64(out)

    def oracle(self, seqs=None, scale=None):
        """fp64 reference (and the rows of the output it covers) for sequences `seqs`."""
        c = self.case
        if seqs is None:
            seqs = np.arange(c.num_seqs)
        rows = np.concatenate([np.arange(c.q_indptr[s], c.q_indptr[s + 1]) for s in seqs])
        q_lens = c.q_indptr[seqs + 1] - c.q_indptr[seqs]
        sub = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
        kc, vc, ks, vs = self.pools
        ref, _ = oracle.attention_int8(c.q[rows], kc, vc, ks, vs, c.block_table[seqs],
                                       c.context_lens[seqs], sub, scale=scale, num_threads=16)
        return ref, rows


@pytest.mark.parametrize("P", [16, 32, 64])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("D", [128, 64])
def test_int8_append_ragged(P, G, D):
    """Ragged contexts and chunk lengths: several 128-position blocks, several tile pairs
    per (sequence, kv head), a ragged last block and a ragged last tile; head_dim 128 and 64
    (64-byte code rows, one-half operands)."""
    case = build_case(500 + P + G + D, name="int8-append", page_size=P, q_heads=2 * G,
                      kv_heads=2, head_dim=D,
                      context_lens=lambda rng: rng.integers(1, 700, size=20),
                      q_lens=lambda ctx: np.minimum(ctx, 1 + (ctx * 7) % 181))
    run = Int8AppendRun(case)
    ref, rows = run.oracle()
    for dtype in (torch.float32, torch.bfloat16):
        assert_close_out(run.attend(dtype)[rows], ref, f"INT8 append P={P} G={G}", dtype)


def test_int8_append_edges():
    """ctx == q_len (no prefix), q_len == 1 (decode through append), chunks that end exactly
    on a block or tile boundary, and one long chunk (many tile pairs)."""
    ctx = np.array([1, 2, 17, 64, 65, 128, 129, 256, 300, 5, 640, 1000])
    qlen = np.array([1, 2, 17, 64, 1, 128, 1, 64, 300, 5, 1, 512])
    case = build_case(78, name="int8-edges", page_size=16, q_heads=8, kv_heads=2, head_dim=128,
                      context_lens=lambda rng: ctx, q_lens=lambda c: qlen)
    run = Int8AppendRun(case)
    ref, rows = run.oracle()
    assert_attention_close(run.attend()[rows], ref, "INT8 append edges")
    # a custom softmax scale reaches the kernel
    ref2, _ = run.oracle(scale=0.05)
    assert_attention_close(run.attend(scale=0.05)[rows], ref2, "INT8 append scale 0.05")


def test_int8_append_of_one_token_matches_int8_decode():
    case = build_case(79, name="int8-one", page_size=16, q_heads=8, kv_heads=2, head_dim=128,
                      context_lens=lambda rng: rng.integers(1, 900, size=16),
                      q_lens=lambda ctx: np.ones_like(ctx))
    run = Int8AppendRun(case)
    got = run.attend()
    out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, device="cuda")
    kvc.kvc_decode_int8(out, run.q, *run.dev, run.bt, run.ctx, case.max_ctx, num_splits=1)
    assert np.abs(got - out_to_f64(out)).max() < 2e-3


@pytest.mark.parametrize("P", [16, 64])
def test_int8_append_rewind_workload_sampled(P):
    """The rewind-append workload (1,000 documents of 300 cached positions, 50 new tokens,
    32 / 8 heads) on INT8 pages, checked on sampled documents."""
    case = config_case(4, page_size=P)
    run = Int8AppendRun(case)
    got = run.attend(torch.bfloat16)
    seqs = sample_seqs(case.num_seqs, 40, seed=P)
    ref, rows = run.oracle(seqs)
    assert_close_out(got[rows], ref, f"INT8 rewind append P={P}", torch.bfloat16)


@pytest.mark.parametrize("P", [16, 64])
def test_int8_append_rewind_workload_f32_every_document(P):
    """The rewind-append workload with fp32 output: all 1,000 documents, held to the plain
    attention tolerance (no allowance for output rounding)."""
    case = config_case(4, page_size=P)
    run = Int8AppendRun(case)
    got = run.attend(torch.float32)
    ref, rows = run.oracle()
    assert_attention_close(got[rows], ref, f"INT8 rewind append P={P}, fp32, every document")


def test_int8_append_single_position_is_its_stored_vector():
    case = build_case(80, name="int8-single", page_size=16, q_heads=4, kv_heads=2,
                      head_dim=128, context_lens=lambda rng: np.array([1, 1]),
                      q_lens=lambda ctx: np.ones_like(ctx))
    run = Int8AppendRun(case)
    got = run.attend()
    kc, vc, ks, vs = run.pools
    for s in range(2):
        page, off = divmod(oracle.slot_of_position(case.block_table, s, 0, 16), 16)
        for h in range(case.q_heads):
            g = h // 2
            want = vs[page, g, off] * vc[page, off, g].astype(np.float64)
            # probability 1 times the value scale enters the PV product as fp16
            np.testing.assert_allclose(got[s, h], want, rtol=2.0 ** -10, atol=1e-6)


def test_int8_append_head_dim_64_edges():
    """head_dim 64: no prefix, one-token chunks, chunks ending on block and tile boundaries,
    a long chunk, and one-position contexts (the output is the stored vector's value)."""
    ctx = np.array([1, 2, 17, 64, 65, 128, 129, 256, 300, 5, 640, 1000, 1])
    qlen = np.array([1, 2, 17, 64, 1, 128, 1, 64, 300, 5, 1, 512, 1])
    case = build_case(82, name="int8-edges-d64", page_size=16, q_heads=8, kv_heads=2,
                      head_dim=64, context_lens=lambda rng: ctx, q_lens=lambda c: qlen)
    run = Int8AppendRun(case)
    ref, rows = run.oracle()
    assert_attention_close(run.attend()[rows], ref, "INT8 append edges D=64")


def test_int8_append_flags_a_value_scale_beyond_fp16_range():
    """A value scale above 4000 (|v| above 5.08e5) cannot enter the fp16 PV product: the
    device error word says so (bit 11) instead of the output silently overflowing."""
    case = build_case(81, name="int8-range", page_size=16, q_heads=4, kv_heads=2,
                      head_dim=128, context_lens=lambda rng: np.array([40, 3]),
                      q_lens=lambda ctx: np.ones_like(ctx))
    run = Int8AppendRun(case)
    assert kvc.kvc_device_errors() == 0
    page, off = divmod(oracle.slot_of_position(case.block_table, 0, 5, 16), 16)
    run.dev[3][page, 1, off] = 5000.0
    c = case
    out = torch.empty(c.num_tokens, c.q_heads, c.head_dim, device="cuda")
    kvc.kvc_append_int8(out, run.q, *run.dev, run.bt, run.ind, run.ctx, c.max_q_len, c.max_ctx)
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 1 << 11
    run.dev[3][page, 1, off] = 4000.0
    kvc.kvc_append_int8(out, run.q, *run.dev, run.bt, run.ind, run.ctx, c.max_q_len, c.max_ctx)
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
