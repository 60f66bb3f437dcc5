"""Fused quantised store + decode over INT8 pages (kvc_decode_int8_store) on the GPU
(TileInfer.jl "KV cache", "INT8 cache": a vector is quantised once, when it is written).

Codes and scales end exactly as the oracle's INT8 store of the new tokens at kvc_slot_mapping's
slots leaves them (over the whole pools; slots that hold no position keep their random codes
and NaN scales), and the output is bit for bit what the separate slot mapping +
kvc_store_int8 + kvc_decode_int8 give, within the attention tolerance of the oracle's fp64
attention over scale * code."""
import numpy as np
import pytest
import torch

import pagedattention_kvc_store_gb300 as kvc
from harness import assert_attention_close, int8_pages, out_to_f64, sample_seqs
from oracle import oracle
from test_gpu_int8 import oracle_int8, run_int8
from workloads import build_case, config_case
from workloads.device import bf16_tensor, i32_tensor

pytestmark = pytest.mark.gpu


def fused_int8(case, out_dtype=torch.float32, num_splits=0, host=False, ctx_override=None):
    kc, vc, ks, vs = (torch.from_numpy(a).cuda() for a in int8_pages(case))
    ctx_np = case.context_lens if ctx_override is None else ctx_override
    args = [bf16_tensor(case.q, "cuda"), bf16_tensor(case.k_new, "cuda"),
            bf16_tensor(case.v_new, "cuda"), i32_tensor(case.block_table, "cuda"),
            i32_tensor(ctx_np, "cuda")]
    out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, dtype=out_dtype,
                      device="cuda")
    if host:
        args = [t.cpu().pin_memory() for t in args]
        out = torch.empty(tuple(out.shape), dtype=out_dtype).pin_memory()
    q, kn, vn, bt, ctx = args
    pool = kvc.int8_pool_desc(kc)
    _, _, ws = kvc.kvc_decode_int8_plan(case.num_seqs, case.q_heads, pool, case.max_ctx,
                                        num_splits)
    work = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    kvc.kvc_decode_int8_store(out, q, kn, vn, kc, vc, ks, vs, bt, ctx, case.max_ctx,
                              num_splits=num_splits, workspace=work)
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
    return out.cpu(), tuple(t.cpu().numpy() for t in (kc, vc, ks, vs))


def assert_pools_equal(got, ref, what):
    for name, g, r in zip(("K codes", "V codes", "K scales", "V scales"), got, ref):
        if g.dtype == np.int8:
            assert np.array_equal(g, r), f"{what}: {name} differ from the oracle's store"
        else:
            assert np.array_equal(np.isnan(g), np.isnan(r)), f"{what}: {name} NaN pattern"
            assert np.array_equal(g[~np.isnan(r)], r[~np.isnan(r)]), f"{what}: {name} differ"


@pytest.mark.parametrize("num_splits", [1, 0, 5])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_batched_decode_int8_store(num_splits, out_dtype):
    """The batched-decode workload (64 sequences, ctx U[512, 4096], 32/8 heads, D 128, P 16)."""
    case = config_case(2)
    out, pools = fused_int8(case, out_dtype, num_splits)
    sep, ref_pools = run_int8(case, num_splits=num_splits, out_dtype=out_dtype)
    assert_pools_equal(pools, ref_pools, "batched")
    assert torch.equal(out, sep.cpu()), "fused output differs from the separate calls'"
    seqs = sample_seqs(case.num_seqs, 10)
    assert_attention_close(out_to_f64(out)[seqs], oracle_int8(case, ref_pools, seqs),
                           f"decode_int8_store splits={num_splits}")


@pytest.mark.parametrize("P", [16, 32, 64])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("D", [128, 64])
def test_edges(P, G, D):
    """One-position contexts and newest positions at the first / last offset of a page, with
    one, three and the planned number of splits, at head_dim 128 and 64."""
    ctx = np.array([1, 2, P - 1, P, P + 1, 2 * P, 3 * P - 1, 5 * P + 7, 64, 65, 700])
    case = build_case(900 + P + G + D, name="int8-decode-store-edges", page_size=P,
                      q_heads=2 * G, kv_heads=2, head_dim=D, context_lens=lambda rng: ctx,
                      q_lens=lambda c: np.minimum(c, 1))
    for splits in (1, 3, 0):
        out, pools = fused_int8(case, num_splits=splits)
        sep, ref_pools = run_int8(case, num_splits=splits)
        assert_pools_equal(pools, ref_pools, f"P={P} G={G} splits={splits}")
        assert torch.equal(out, sep.cpu()), (P, G, splits)
        assert_attention_close(out_to_f64(out), oracle_int8(case, ref_pools),
                               f"decode_int8_store edges P={P} G={G} splits={splits}")


def test_host_fed_equals_device_fed():
    """q, k_new, v_new, the tables and out in pinned host memory give the same bytes."""
    case = config_case(2, num_seqs=24)
    dev = fused_int8(case, torch.bfloat16)
    host = fused_int8(case, torch.bfloat16, host=True)
    assert torch.equal(dev[0], host[0])
    assert_pools_equal(host[1], dev[1], "host-fed")


def test_empty_context_stores_nothing():
    """A sequence with context length 0 has no slot for its token: nothing is stored for it
    and its output is 0 (one split, and several with the merge)."""
    case = config_case(2, num_seqs=8)
    ctx = case.context_lens.copy()
    ctx[2] = 0
    ref = list(int8_pages(case))
    slots = np.array([oracle.slot_of_position(case.block_table, s, int(c) - 1, case.page_size)
                      if c > 0 else -1 for s, c in enumerate(ctx)], dtype=np.int64)
    keep = slots >= 0
    oracle.store_int8(*ref, case.k_new[keep], case.v_new[keep], slots[keep])
    for splits in (1, 2):
        out, pools = fused_int8(case, num_splits=splits, ctx_override=ctx)
        assert_pools_equal(pools, ref, f"empty context, splits={splits}")
        assert not out[2].any()
        assert out.isfinite().all()


def test_null_new_rows_are_refused():
    case = config_case(2, num_seqs=4)
    kc, vc, ks, vs = (torch.from_numpy(a).cuda() for a in int8_pages(case))
    out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, device="cuda")
    q = bf16_tensor(case.q, "cuda")
    bt, ctx = i32_tensor(case.block_table, "cuda"), i32_tensor(case.context_lens, "cuda")
    st = kvc.lib().kvc_decode_int8_store(
        out.data_ptr(), kvc.KVC_F32, q.data_ptr(), None, None, kc.data_ptr(), vc.data_ptr(),
        ks.data_ptr(), vs.data_ptr(), kvc.int8_pool_desc(kc), bt.data_ptr(),
        int(bt.shape[1]), ctx.data_ptr(), case.num_seqs, case.max_ctx, case.q_heads, 0.0, 1,
        None, 0, None)
    assert st != 0


def test_decode_int8_reads_pinned_host_memory():
    """kvc_decode_int8 alone: q, the tables and out in pinned host memory give the device-fed
    bytes (the pools hold the new tokens already, stored by the fused call)."""
    case = config_case(2, num_seqs=16)
    dev_out, pools = fused_int8(case, torch.bfloat16, num_splits=3)
    kc, vc, ks, vs = (torch.from_numpy(a).cuda() for a in pools)
    args = [bf16_tensor(case.q, "cuda"), i32_tensor(case.block_table, "cuda"),
            i32_tensor(case.context_lens, "cuda")]
    q, bt, ctx = (t.cpu().pin_memory() for t in args)
    out = torch.empty(tuple(dev_out.shape), dtype=torch.bfloat16).pin_memory()
    _, _, ws = kvc.kvc_decode_int8_plan(case.num_seqs, case.q_heads, kvc.int8_pool_desc(kc),
                                        case.max_ctx, 3)
    kvc.kvc_decode_int8(out, q, kc, vc, ks, vs, bt, ctx, case.max_ctx, num_splits=3,
                        workspace=torch.empty(ws, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
    assert torch.equal(out, dev_out)


def test_decode_int8_refuses_pageable_host_out():
    """A host pointer the device cannot reach at that address is refused before anything is
    enqueued (the C entry point, bypassing the binding's own check)."""
    import ctypes
    case = config_case(2, num_seqs=4)
    kc, vc, ks, vs = (torch.from_numpy(a).cuda() for a in int8_pages(case))
    q = bf16_tensor(case.q, "cuda")
    bt, ctx = i32_tensor(case.block_table, "cuda"), i32_tensor(case.context_lens, "cuda")
    host = np.zeros(case.num_seqs * case.q_heads * case.head_dim + 8, dtype=np.float32)
    addr = (host.ctypes.data + 15) // 16 * 16
    st = kvc.lib().kvc_decode_int8(
        ctypes.c_void_p(addr), kvc.KVC_F32, q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
        ks.data_ptr(), vs.data_ptr(), kvc.int8_pool_desc(kc), bt.data_ptr(), int(bt.shape[1]),
        ctx.data_ptr(), case.num_seqs, case.max_ctx, case.q_heads, 0.0, 1, None, 0, None)
    assert st == 1 and b"pinned host" in kvc.lib().kvc_last_error()
    torch.cuda.synchronize()
    assert not host.any()
