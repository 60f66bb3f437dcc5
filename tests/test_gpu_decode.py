"""GPU parity of paged decode (split-K and merge) against the fp64 oracle."""
import ctypes

import numpy as np
import pytest
import torch

import pagedattention_kvc_store_gb300 as kvc
from harness import (GpuRun, OracleRun, THREADS, assert_attention_close, out_to_f64,
                     sample_seqs)
from oracle import oracle
from workloads import build_case, config_case, f32_from_bf16
from workloads.device import bf16_bits_of, bf16_tensor

pytestmark = pytest.mark.gpu


def _decode_case(seed, S, ctx_lo, ctx_hi, P, Hq, Hkv, D, ctx=None):
    return build_case(seed, name="decode", page_size=P, q_heads=Hq, kv_heads=Hkv, head_dim=D,
                      context_lens=(lambda rng: np.array(ctx)) if ctx is not None else
                      (lambda rng: rng.integers(ctx_lo, ctx_hi + 1, size=S)),
                      q_lens=np.ones_like)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("num_splits", [1, 2, 0])
def test_tiny_decode(out_dtype, num_splits):
    case = config_case(1)
    g = GpuRun(case, decode=True)
    g.store()
    out = g.attend(out_dtype, num_splits)
    ref, _ = OracleRun(case).attention()
    assert_attention_close(out_to_f64(out), ref, "tiny decode")
    # ctx = 1: the output is the stored value itself, bit for bit
    v0 = f32_from_bf16(case.v_new[0])           # [Hkv, D]
    got = out[0].float().cpu().numpy()
    for h in range(case.q_heads):
        np.testing.assert_array_equal(got[h], v0[h // 2])


@pytest.mark.parametrize("num_splits", [1, 2, 7, 0])
def test_batched_decode_full_size(num_splits):
    case = config_case(2)
    g = GpuRun(case, decode=True)
    g.store()
    out = g.attend(torch.bfloat16, num_splits)
    ref, _ = OracleRun(case).attention()
    assert_attention_close(out_to_f64(out), ref, f"batched decode, splits={num_splits}")


def test_split_partials_match_the_oracle_windows():
    case = config_case(2, num_seqs=12)
    g = GpuRun(case, decode=True)
    g.store()
    g.attend(torch.float32, num_splits=3)
    pool = kvc.pool_desc(g.d.k_pool)
    splits, chunk, ws = kvc.kvc_decode_plan(case.num_seqs, case.q_heads, pool, case.max_ctx, 3)
    assert splits == 3
    rows = case.num_seqs * case.q_heads
    o_bytes = rows * splits * case.head_dim * 4
    lse_off = -(-o_bytes // 256) * 256
    wsb = g.workspace.cpu().numpy()
    part_o = wsb[:o_bytes].view(np.float32).reshape(case.num_seqs, case.q_heads, splits, -1)
    part_lse = wsb[lse_off: lse_off + rows * splits * 4].view(np.float32).reshape(
        case.num_seqs, case.q_heads, splits)
    o = OracleRun(case)
    for j in range(splits):
        lo = np.full(case.num_seqs, j * chunk, np.int32)
        hi = np.full(case.num_seqs, (j + 1) * chunk, np.int32)
        ref_o, ref_l = oracle.attention(case.q, o.k_pool, o.v_pool, case.block_table,
                                        case.context_lens, case.q_indptr, key_lo=lo, key_hi=hi,
                                        num_threads=THREADS)
        empty = np.isneginf(ref_l)
        assert np.array_equal(np.isneginf(part_lse[:, :, j]), empty)
        live = ~empty
        assert_attention_close(part_o[:, :, j][live].astype(np.float64), ref_o[live],
                               f"partial {j}", max_abs=2e-3, mean_abs=2e-4)
        np.testing.assert_allclose(part_lse[:, :, j][live], ref_l[live], rtol=0, atol=2e-3)


def test_merge_against_oracle_merge():
    rng = np.random.default_rng(3)
    rows, splits, D = 77, 9, 128
    po = rng.standard_normal((rows, splits, D)).astype(np.float32)
    pl = (rng.standard_normal((rows, splits)) * 3).astype(np.float32)
    pl[rng.random((rows, splits)) < 0.3] = -np.inf
    pl[5] = -np.inf                                  # a row with no key at all
    po[np.isneginf(pl)] = np.nan                      # never read
    out = torch.empty(rows, D, dtype=torch.float32, device="cuda")
    lse = torch.empty(rows, dtype=torch.float32, device="cuda")
    kvc.kvc_merge(out, torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda(), lse)
    ref, ref_lse = oracle.merge(po.astype(np.float64), pl.astype(np.float64))
    got = out.cpu().numpy()
    assert np.isfinite(got).all() and (got[5] == 0).all()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-5)
    gl = lse.cpu().numpy()
    assert np.isneginf(gl[5])
    np.testing.assert_allclose(gl[np.isfinite(ref_lse)], ref_lse[np.isfinite(ref_lse)],
                               rtol=0, atol=1e-5)


def test_shared_prefix_decode_full_size():
    case = config_case(3)
    g = GpuRun(case, decode=True)
    g.store()
    out = g.attend(torch.bfloat16, 0)
    ref, _ = OracleRun(case).attention()
    assert_attention_close(out_to_f64(out), ref, "shared-prefix decode")


@pytest.mark.slow
def test_long_context_decode_full_size():
    case = config_case(5)
    g = GpuRun(case, decode=True)
    g.store()
    out = g.attend(torch.bfloat16, 0)
    ref, _ = OracleRun(case).attention()
    assert_attention_close(out_to_f64(out), ref, "long decode")


@pytest.mark.parametrize("P,Hq,Hkv,D", [(16, 8, 8, 64), (32, 16, 8, 128), (64, 16, 2, 64),
                                        (16, 16, 2, 128), (32, 4, 4, 128), (64, 64, 8, 64)])
def test_decode_shapes(P, Hq, Hkv, D):
    case = _decode_case(P * 7 + Hq + D, 13, 1, 700, P, Hq, Hkv, D)
    for splits in (1, 0, 5):
        g = GpuRun(case, decode=True)
        g.store()
        out = g.attend(torch.float32, splits)
        ref, _ = OracleRun(case).attention()
        assert_attention_close(out_to_f64(out), ref, f"{P},{Hq},{Hkv},{D} splits={splits}")


def test_edge_lengths_and_empty_sequences():
    ctx = [0, 1, 15, 16, 17, 63, 64, 65, 127, 128, 129, 1000, 0]
    case = _decode_case(9, len(ctx), 0, 0, 16, 8, 2, 128, ctx=ctx)
    # sequences with ctx 0 have no new token to store; their slot must be skipped
    for splits in (1, 3, 0):
        g = GpuRun(case, decode=True)
        g.store()
        out = g.attend(torch.float32, splits)
        got = out_to_f64(out)
        assert (got[0] == 0).all() and (got[-1] == 0).all()
        ref, _ = OracleRun(case).attention()
        assert_attention_close(got, ref, f"edge lengths, splits={splits}")


def test_empty_batch_is_a_no_op():
    case = config_case(1)
    g = GpuRun(case, decode=True)
    out = torch.full((0, 4, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    kvc.kvc_decode(out, g.d.q[:0], g.d.k_pool, g.d.v_pool, g.d.block_table[:0],
                   g.d.context_lens[:0], 0)
    torch.cuda.synchronize()


def test_physical_placement_gives_identical_bits():
    case = config_case(2, num_seqs=16)
    g1 = GpuRun(case, decode=True)
    g1.store()
    out1 = g1.attend(torch.bfloat16, 0)
    relabel = np.random.default_rng(1).permutation(case.num_pages)
    case2 = config_case(2, num_seqs=16)
    case2.k_pool[relabel] = case.k_pool
    case2.v_pool[relabel] = case.v_pool
    held = np.zeros_like(case.block_table, dtype=bool)
    for s, n in enumerate(case.context_lens):
        held[s, : -(-int(n) // case.page_size)] = True
    case2.block_table = np.where(held, relabel[case.block_table], 0).astype(np.int32)
    g2 = GpuRun(case2, decode=True)
    g2.store()
    out2 = g2.attend(torch.bfloat16, 0)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_no_device_errors_were_raised():
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0


@pytest.mark.parametrize("num_splits", [1, 0])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_decode_into_pinned_host_out(num_splits, out_dtype):
    """out may be pinned host memory: the kernel that finishes each row (the decode itself
    with one split, the merge otherwise) writes it there, bit for bit what a device out
    receives; kvc_merge accepts a pinned host out the same way."""
    case = config_case(2, num_seqs=16)
    g = GpuRun(case, decode=True)
    g.store()
    dev_out = g.attend(out_dtype, num_splits)
    host_out = torch.full(tuple(dev_out.shape), float("nan"), dtype=out_dtype).pin_memory()
    c, d = g.case, g.d
    kvc.kvc_decode(host_out, d.q, d.k_pool, d.v_pool, d.block_table, d.context_lens, c.max_ctx,
                   num_splits=num_splits, workspace=g.workspace)
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
    assert torch.equal(host_out, dev_out.cpu())


def test_merge_into_pinned_host_out():
    rng = np.random.default_rng(3)
    rows, splits, D = 37, 5, 128
    po = torch.tensor(rng.standard_normal((rows, splits, D)), dtype=torch.float32, device="cuda")
    lse = torch.tensor(rng.standard_normal((rows, splits)), dtype=torch.float32, device="cuda")
    lse[3, :] = float("-inf")   # a row with no key
    dev_out = torch.empty(rows, D, dtype=torch.bfloat16, device="cuda")
    host_out = torch.empty(rows, D, dtype=torch.bfloat16).pin_memory()
    kvc.kvc_merge(dev_out, po, lse)
    kvc.kvc_merge(host_out, po, lse)
    torch.cuda.synchronize()
    assert torch.equal(host_out, dev_out.cpu())
    assert not host_out[3].float().any()


def test_decode_refuses_pageable_host_out():
    """A host pointer the device cannot reach at that address is refused before anything is
    enqueued (the C entry point, bypassing the binding's own check)."""
    from pagedattention_kvc_store_gb300.kvc import lib, pool_desc, _ptr
    case = config_case(1)
    g = GpuRun(case, decode=True)
    g.store()
    c, d = g.case, g.d
    host = np.zeros(c.num_seqs * c.q_heads * c.head_dim + 8, dtype=np.float32)
    addr = (host.ctypes.data + 15) // 16 * 16
    st = lib().kvc_decode(ctypes.c_void_p(addr), 1, _ptr(d.q), _ptr(d.k_pool), _ptr(d.v_pool),
                          pool_desc(d.k_pool), _ptr(d.block_table), int(d.block_table.shape[1]),
                          _ptr(d.context_lens), c.num_seqs, c.max_ctx, c.q_heads, 0.0, 1, None,
                          0, None)
    assert st == 1 and b"pinned host" in lib().kvc_last_error()
    torch.cuda.synchronize()
    assert not host.any()


@pytest.mark.parametrize("num_splits", [1, 0])
def test_decode_reads_pinned_host_inputs(num_splits):
    """q, block_table and context_lens may sit in pinned host memory (with the output too):
    the kernels read them across the host link and give the device-fed result bit for bit."""
    case = config_case(2, num_seqs=24)
    g = GpuRun(case, decode=True)
    g.store()
    dev_out = g.attend(torch.bfloat16, num_splits)
    d = g.d
    hq, hbt, hctx = (t.cpu().pin_memory() for t in (d.q, d.block_table, d.context_lens))
    host_out = torch.empty(tuple(dev_out.shape), dtype=torch.bfloat16).pin_memory()
    kvc.kvc_decode(host_out, hq, d.k_pool, d.v_pool, hbt, hctx, case.max_ctx,
                   num_splits=num_splits, workspace=g.workspace)
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
    assert torch.equal(host_out, dev_out.cpu())
