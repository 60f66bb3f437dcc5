"""HND pools on the GPU (TileInfer.jl "KV cache", "Pages and block tables": one contiguous
[page_size][head_dim] block per (page, kv head)).  The same seeded caches as the NHD tests,
transposed into the HND layout: the store is bit-exact against the oracle's HND store, and
decode, append and shared-prefix decode agree with the oracle over the HND pools."""
import numpy as np
import pytest
import torch

import pagedattention_kvc_store_gb300 as kvc
from harness import assert_attention_close, out_to_f64, sample_seqs
from oracle import oracle
from workloads import build_case, config_case
from workloads.device import bf16_bits_of, bf16_tensor, i32_tensor

pytestmark = pytest.mark.gpu


def _hnd_run(case, decode):
    """Store the case's new tokens into HND pools on the GPU and in the oracle."""
    k_h, v_h = oracle.nhd_to_hnd(case.k_pool), oracle.nhd_to_hnd(case.v_pool)
    kd, vd = bf16_tensor(k_h, "cuda"), bf16_tensor(v_h, "cuda")
    bt, ctx = i32_tensor(case.block_table, "cuda"), i32_tensor(case.context_lens, "cuda")
    ind = i32_tensor(case.q_indptr, "cuda")
    slots = torch.empty(case.num_tokens, dtype=torch.int32, device="cuda")
    kvc.kvc_slot_mapping(slots, bt, ctx, None if decode else ind, case.page_size,
                         max_q_len=case.max_q_len)
    kvc.kvc_store(kd, vd, bf16_tensor(case.k_new, "cuda"), bf16_tensor(case.v_new, "cuda"),
                  slots, layout="hnd")
    oracle.store(k_h, v_h, case.k_new, case.v_new, slots.cpu().numpy().astype(np.int64),
                 layout="hnd")
    assert np.array_equal(bf16_bits_of(kd), k_h), "K pool (HND) differs from the oracle's"
    assert np.array_equal(bf16_bits_of(vd), v_h), "V pool (HND) differs from the oracle's"
    return kd, vd, bt, ctx, ind, k_h, v_h


@pytest.mark.parametrize("P", [16, 32, 64])
@pytest.mark.parametrize("splits", [1, 0])
def test_hnd_decode(P, splits):
    case = build_case(900 + P, name="hnd-decode", page_size=P, q_heads=8, kv_heads=2,
                      head_dim=128, context_lens=lambda rng: rng.integers(1, 900, size=20),
                      q_lens=lambda ctx: np.ones_like(ctx))
    kd, vd, bt, ctx, _, k_h, v_h = _hnd_run(case, decode=True)
    out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, dtype=torch.float32,
                      device="cuda")
    pool = kvc.pool_desc(kd, "hnd")
    _, _, ws = kvc.kvc_decode_plan(case.num_seqs, case.q_heads, pool, case.max_ctx, splits)
    work = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    kvc.kvc_decode(out, bf16_tensor(case.q, "cuda"), kd, vd, bt, ctx, case.max_ctx,
                   num_splits=splits, workspace=work, layout="hnd")
    ref, _ = oracle.attention(case.q, k_h, v_h, case.block_table, case.context_lens,
                              case.q_indptr, layout="hnd", num_threads=16)
    assert_attention_close(out_to_f64(out), ref, f"HND decode P={P}")
    assert kvc.kvc_device_errors() == 0


def test_hnd_tiny_decode_head_dim_64():
    case = config_case(1)
    kd, vd, bt, ctx, _, k_h, v_h = _hnd_run(case, decode=True)
    out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, dtype=torch.float32,
                      device="cuda")
    kvc.kvc_decode(out, bf16_tensor(case.q, "cuda"), kd, vd, bt, ctx, case.max_ctx,
                   num_splits=1, layout="hnd")
    ref, _ = oracle.attention(case.q, k_h, v_h, case.block_table, case.context_lens,
                              case.q_indptr, layout="hnd")
    assert_attention_close(out_to_f64(out), ref, "HND tiny decode")


@pytest.mark.parametrize("P", [16, 64])
def test_hnd_append_rewind_sample(P):
    """The rewind-append workload (1,000 x 50 over 300) on HND pools, sampled documents."""
    case = config_case(4, page_size=P)
    kd, vd, bt, ctx, ind, k_h, v_h = _hnd_run(case, decode=False)
    out = torch.empty(case.num_tokens, case.q_heads, case.head_dim, dtype=torch.bfloat16,
                      device="cuda")
    kvc.kvc_append(out, bf16_tensor(case.q, "cuda"), kd, vd, bt, ind, ctx, case.max_q_len,
                   case.max_ctx, layout="hnd")
    seqs = sample_seqs(case.num_seqs, 40, seed=3)
    rows = np.concatenate([np.arange(case.q_indptr[s], case.q_indptr[s + 1]) for s in seqs])
    q_lens = case.q_indptr[seqs + 1] - case.q_indptr[seqs]
    sub_ind = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    ref, _ = oracle.attention(case.q[rows], k_h, v_h, case.block_table[seqs],
                              case.context_lens[seqs], sub_ind, layout="hnd", num_threads=16)
    assert_attention_close(out_to_f64(out)[rows], ref, f"HND append P={P}")
    assert kvc.kvc_device_errors() == 0


def test_hnd_shared_prefix_decode():
    case = config_case(3)
    kd, vd, bt, ctx, _, k_h, v_h = _hnd_run(case, decode=True)
    out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, dtype=torch.float32,
                      device="cuda")
    indptr = np.arange(0, case.num_seqs + 1, 8, dtype=np.int32)
    prefix = np.full(len(case.groups), case.shared_positions, np.int32)
    gi, gs, gp = (i32_tensor(indptr, "cuda"), i32_tensor(np.concatenate(case.groups), "cuda"),
                  i32_tensor(prefix, "cuda"))
    pool = kvc.pool_desc(kd, "hnd")
    ws = kvc.kvc_decode_shared_prefix_plan(case.num_seqs, case.q_heads, pool, case.max_ctx,
                                           len(case.groups), int(prefix.max()))
    work = torch.empty(ws, dtype=torch.uint8, device="cuda")
    kvc.kvc_decode_shared_prefix(out, bf16_tensor(case.q, "cuda"), kd, vd, bt, ctx, case.max_ctx,
                                 gi, gs, gp, 8, int(prefix.max()), work, layout="hnd")
    seqs = sample_seqs(case.num_seqs, 24, seed=5)
    ind = np.arange(len(seqs) + 1, dtype=np.int32)
    ref, _ = oracle.attention(case.q[seqs], k_h, v_h, case.block_table[seqs],
                              case.context_lens[seqs], ind, layout="hnd", num_threads=16)
    assert_attention_close(out_to_f64(out)[seqs], ref, "HND shared-prefix decode")
    assert kvc.kvc_device_errors() == 0


def test_int8_refuses_hnd():
    pool = kvc.PoolDesc(8, 16, 2, 128, kvc.KVC_HND)
    k = torch.zeros(8, 16, 2, 128, dtype=torch.int8, device="cuda")
    s = torch.zeros(8, 2, 16, device="cuda")
    new = torch.zeros(1, 2, 128, dtype=torch.bfloat16, device="cuda")
    slots = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = kvc.lib().kvc_store_int8(k.data_ptr(), k.data_ptr(), s.data_ptr(), s.data_ptr(), pool,
                                  new.data_ptr(), new.data_ptr(), slots.data_ptr(), 1, None)
    assert kvc.kvc.STATUS[st] == "KVC_ERR_UNSUPPORTED"
