"""Fused store + decode (kvc_decode_store) on the GPU: the pools end exactly as kvc_store with
kvc_slot_mapping's slots leaves them (bit-exact against the oracle's store, over the whole
pool), and the output is bit for bit what the separate slot mapping + store + decode give."""
import numpy as np
import pytest
import torch

import pagedattention_kvc_store_gb300 as kvc
from harness import GpuRun, OracleRun, assert_attention_close, out_to_f64
from oracle import oracle
from workloads import build_case, config_case
from workloads.device import bf16_bits_of, bf16_tensor, to_device

pytestmark = pytest.mark.gpu


def fused(case, out_dtype, num_splits, layout="nhd", host=False):
    d = to_device(case)
    kp, vp = d.k_pool, d.v_pool
    if layout == "hnd":
        kp = bf16_tensor(oracle.nhd_to_hnd(case.k_pool), "cuda")
        vp = bf16_tensor(oracle.nhd_to_hnd(case.v_pool), "cuda")
    pool = kvc.pool_desc(kp, layout)
    _, _, ws = kvc.kvc_decode_plan(case.num_seqs, case.q_heads, pool, case.max_ctx, num_splits)
    work = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    args = [d.q, d.k_new, d.v_new, d.block_table, d.context_lens]
    out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, dtype=out_dtype,
                      device="cuda")
    if host:
        args = [t.cpu().pin_memory() for t in args]
        out = torch.empty(tuple(out.shape), dtype=out_dtype).pin_memory()
    q, kn, vn, bt, ctx = args
    kvc.kvc_decode_store(out, q, kn, vn, kp, vp, bt, ctx, case.max_ctx, num_splits=num_splits,
                         workspace=work, layout=layout)
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
    return out.cpu(), bf16_bits_of(kp), bf16_bits_of(vp)


def separate(case, out_dtype, num_splits):
    g = GpuRun(case, decode=True)
    g.store()
    out = g.attend(out_dtype, num_splits)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("num_splits", [1, 0, 7])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_batched_decode_store(num_splits, out_dtype):
    case = config_case(2)
    out, kb, vb = fused(case, out_dtype, num_splits)
    o = OracleRun(case)
    assert np.array_equal(kb, o.k_pool), "K pool differs from the oracle's store"
    assert np.array_equal(vb, o.v_pool), "V pool differs from the oracle's store"
    assert torch.equal(out, separate(case, out_dtype, num_splits))
    ref, _ = o.attention()
    assert_attention_close(out_to_f64(out), ref, "decode_store")


def test_edges_and_hnd():
    """One-position contexts, a newest position at the first / last offset of its page,
    several page sizes; HND pools."""
    for P, Hq, Hkv, D in ((16, 32, 8, 128), (32, 8, 2, 64), (64, 16, 8, 128), (16, 8, 8, 128),
                          (32, 64, 8, 64)):
        ctx = np.array([1, 2, P, P + 1, 2 * P, 3 * P - 1, 5 * P + 7, 700])
        case = build_case(P + D + Hq, name="decode-store-edges", page_size=P, q_heads=Hq,
                          kv_heads=Hkv, head_dim=D, context_lens=lambda rng: ctx,
                          q_lens=lambda c: np.minimum(c, 1))
        o = OracleRun(case)
        for layout in ("nhd", "hnd"):
            out, kb, vb = fused(case, torch.float32, 0, layout=layout)
            k_ref, v_ref = o.k_pool, o.v_pool
            if layout == "hnd":
                k_ref, v_ref = oracle.nhd_to_hnd(k_ref), oracle.nhd_to_hnd(v_ref)
            assert np.array_equal(kb, k_ref) and np.array_equal(vb, v_ref), (P, layout)
            ref, _ = o.attention()
            assert_attention_close(out_to_f64(out), ref, f"decode_store edges {P} {layout}")


def test_host_fed_equals_device_fed():
    case = config_case(2, num_seqs=24)
    dev = fused(case, torch.bfloat16, 0)
    host = fused(case, torch.bfloat16, 0, host=True)
    assert torch.equal(dev[0], host[0])
    assert np.array_equal(dev[1], host[1]) and np.array_equal(dev[2], host[2])


def test_empty_context_stores_nothing():
    """A sequence with context length 0 has no position for its token: nothing is stored for
    it and its output is 0, as with the separate calls (slot -1, skipped)."""
    case = config_case(1)
    d1, d2 = to_device(case), to_device(case)
    for d in (d1, d2):
        d.context_lens[2] = 0
    out1 = torch.empty(case.num_seqs, case.q_heads, case.head_dim, dtype=torch.float32,
                       device="cuda")
    out2 = torch.empty_like(out1)
    kvc.kvc_decode_store(out1, d1.q, d1.k_new, d1.v_new, d1.k_pool, d1.v_pool, d1.block_table,
                         d1.context_lens, case.max_ctx, num_splits=1)
    # with two splits (partials and merge): the empty sequence's output is 0 as well
    pool = kvc.pool_desc(d1.k_pool)
    _, _, ws = kvc.kvc_decode_plan(case.num_seqs, case.q_heads, pool, case.max_ctx, 2)
    out3 = torch.full_like(out1, float("nan"))
    kvc.kvc_decode_store(out3, d1.q, d1.k_new, d1.v_new, d1.k_pool, d1.v_pool, d1.block_table,
                         d1.context_lens, case.max_ctx, num_splits=2,
                         workspace=torch.empty(ws, dtype=torch.uint8, device="cuda"))
    slots = torch.empty(case.num_seqs, dtype=torch.int32, device="cuda")
    kvc.kvc_slot_mapping(slots, d2.block_table, d2.context_lens, None, case.page_size)
    kvc.kvc_store(d2.k_pool, d2.v_pool, d2.k_new, d2.v_new, slots)
    kvc.kvc_decode(out2, d2.q, d2.k_pool, d2.v_pool, d2.block_table, d2.context_lens,
                   case.max_ctx, num_splits=1)
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
    assert int(slots[2].item()) == -1
    assert np.array_equal(bf16_bits_of(d1.k_pool), bf16_bits_of(d2.k_pool))
    assert np.array_equal(bf16_bits_of(d1.v_pool), bf16_bits_of(d2.v_pool))
    assert torch.equal(out1, out2) and not out1[2].any()
    assert not out3[2].any() and (out3 - out1).abs().max().item() < 2e-3


def test_repeated_calls_and_graph_replay():
    """Storing the same new tokens again leaves the pools and the output as they were:
    repeated calls and replays of a captured graph give the same output."""
    case = config_case(2)
    d = to_device(case)
    pool = kvc.pool_desc(d.k_pool)
    sp, _, ws = kvc.kvc_decode_plan(case.num_seqs, case.q_heads, pool, case.max_ctx, 0)
    work = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, dtype=torch.bfloat16,
                      device="cuda")

    def call():
        kvc.kvc_decode_store(out, d.q, d.k_new, d.v_new, d.k_pool, d.v_pool, d.block_table,
                             d.context_lens, case.max_ctx, workspace=work)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    first = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for _ in range(3):
        g.replay()
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
    assert torch.equal(out, first)


def test_host_fed_hnd():
    case = config_case(2, num_seqs=16)
    dev = fused(case, torch.float32, 0, layout="hnd")
    host = fused(case, torch.float32, 0, layout="hnd", host=True)
    assert torch.equal(dev[0], host[0])
    assert np.array_equal(dev[1], host[1]) and np.array_equal(dev[2], host[2])
    o = OracleRun(case)
    assert np.array_equal(dev[1], oracle.nhd_to_hnd(o.k_pool))
