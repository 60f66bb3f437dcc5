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


def _int8_hnd_and_nhd(case):
    """INT8 pools of the case (cached positions quantised by the oracle, NaN scales and random
    codes elsewhere) in both layouts on the GPU, and the new tokens stored into each by
    kvc_store_int8; returns the oracle's pools after its own store (NHD) and both GPU sets."""
    from harness import int8_pages
    kc, vc, ks, vs = int8_pages(case)
    slots = torch.empty(case.num_tokens, dtype=torch.int32, device="cuda")
    bt, ctx = i32_tensor(case.block_table, "cuda"), i32_tensor(case.context_lens, "cuda")
    ind = i32_tensor(case.q_indptr, "cuda")
    kvc.kvc_slot_mapping(slots, bt, ctx, ind, case.page_size, max_q_len=case.max_q_len)
    k_new, v_new = bf16_tensor(case.k_new, "cuda"), bf16_tensor(case.v_new, "cuda")
    sets = {}
    for layout, conv in (("nhd", lambda a: a), ("hnd", oracle.nhd_to_hnd)):
        dev = [torch.from_numpy(np.ascontiguousarray(conv(kc))).cuda(),
               torch.from_numpy(np.ascontiguousarray(conv(vc))).cuda(),
               torch.from_numpy(ks.copy()).cuda(), torch.from_numpy(vs.copy()).cuda()]
        kvc.kvc_store_int8(*dev, k_new, v_new, slots, layout=layout)
        sets[layout] = dev
    oracle.store_int8(kc, vc, ks, vs, case.k_new, case.v_new,
                      slots.cpu().numpy().astype(np.int64))
    torch.cuda.synchronize()
    return (kc, vc, ks, vs), sets, (bt, ctx, ind)


def test_int8_hnd_store_decode_and_append():
    """INT8 pages in the HND layout: kvc_store_int8 writes the oracle's codes (in the HND
    order) and scales, bit for bit; kvc_decode_int8 and kvc_append_int8 over HND pools give
    exactly the NHD pools' outputs (same operands, only the addressing differs) and match the
    oracle's attention."""
    from test_gpu_int8 import oracle_int8
    for P, G in ((16, 4), (64, 8), (32, 1)):
        case = build_case(600 + P + G, name="int8-hnd", page_size=P, q_heads=2 * G,
                          kv_heads=2, head_dim=128,
                          context_lens=lambda rng: rng.integers(1, 600, size=18),
                          q_lens=lambda ctx: np.ones_like(ctx))
        ref_pools, sets, (bt, ctx, _) = _int8_hnd_and_nhd(case)
        kc, vc, ks, vs = ref_pools
        got = [t.cpu().numpy() for t in sets["hnd"]]
        assert np.array_equal(got[0], oracle.nhd_to_hnd(kc)), "HND K codes"
        assert np.array_equal(got[1], oracle.nhd_to_hnd(vc)), "HND V codes"
        for g, r in zip(got[2:], (ks, vs)):
            assert np.array_equal(g, r, equal_nan=True), "HND scales"
        q = bf16_tensor(case.q, "cuda")
        outs = {}
        for layout, dev in sets.items():
            out = torch.empty(case.num_seqs, case.q_heads, 128, device="cuda")
            work = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")
            kvc.kvc_decode_int8(out, q, *dev, bt, ctx, case.max_ctx, num_splits=3,
                                workspace=work, layout=layout)
            outs[layout] = out
        torch.cuda.synchronize()
        assert torch.equal(outs["hnd"], outs["nhd"]), f"INT8 decode HND != NHD (P={P})"
        assert_attention_close(out_to_f64(outs["hnd"]), oracle_int8(case, ref_pools),
                               f"INT8 HND decode P={P}")
    # append (chunks over cached prefixes) on HND pools
    case = build_case(611, name="int8-hnd-append", page_size=16, q_heads=8, kv_heads=2,
                      head_dim=128, context_lens=lambda rng: rng.integers(1, 500, size=14),
                      q_lens=lambda ctx: np.minimum(ctx, 1 + (ctx * 7) % 181))
    ref_pools, sets, (bt, ctx, ind) = _int8_hnd_and_nhd(case)
    q = bf16_tensor(case.q, "cuda")
    outs = {}
    for layout, dev in sets.items():
        out = torch.empty(case.num_tokens, case.q_heads, 128, device="cuda")
        kvc.kvc_append_int8(out, q, *dev, bt, ind, ctx, case.max_q_len, case.max_ctx,
                            layout=layout)
        outs[layout] = out
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
    assert torch.equal(outs["hnd"], outs["nhd"]), "INT8 append HND != NHD"
    kc, vc, ks, vs = ref_pools
    ref, _ = oracle.attention_int8(case.q, kc, vc, ks, vs, case.block_table, case.context_lens,
                                   case.q_indptr, num_threads=16)
    assert_attention_close(out_to_f64(outs["hnd"]), ref, "INT8 HND append")


def test_int8_hnd_decode_store():
    """kvc_decode_int8_store on HND pools: the new tokens' codes land at their HND rows, bit
    for bit, and the output equals the NHD pools' (and the oracle's within tolerance)."""
    from harness import int8_pages
    from test_gpu_int8 import oracle_int8
    case = build_case(612, name="int8-hnd-fused", page_size=16, q_heads=8, kv_heads=2,
                      head_dim=128, context_lens=lambda rng: rng.integers(1, 700, size=16),
                      q_lens=lambda ctx: np.ones_like(ctx))
    kc, vc, ks, vs = int8_pages(case)
    bt, ctx = i32_tensor(case.block_table, "cuda"), i32_tensor(case.context_lens, "cuda")
    q = bf16_tensor(case.q, "cuda")
    k_new, v_new = bf16_tensor(case.k_new, "cuda"), bf16_tensor(case.v_new, "cuda")
    outs, pools = {}, {}
    for layout, conv in (("nhd", lambda a: a), ("hnd", oracle.nhd_to_hnd)):
        dev = [torch.from_numpy(np.ascontiguousarray(conv(kc))).cuda(),
               torch.from_numpy(np.ascontiguousarray(conv(vc))).cuda(),
               torch.from_numpy(ks.copy()).cuda(), torch.from_numpy(vs.copy()).cuda()]
        out = torch.empty(case.num_seqs, case.q_heads, 128, device="cuda")
        work = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")
        kvc.kvc_decode_int8_store(out, q, k_new, v_new, *dev, bt, ctx, case.max_ctx,
                                  num_splits=2, workspace=work, layout=layout)
        outs[layout], pools[layout] = out, dev
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
    slots = oracle.slot_mapping(case.block_table, case.context_lens, case.q_indptr,
                                case.page_size)
    oracle.store_int8(kc, vc, ks, vs, case.k_new, case.v_new, slots)
    assert np.array_equal(pools["hnd"][0].cpu().numpy(), oracle.nhd_to_hnd(kc))
    assert np.array_equal(pools["hnd"][1].cpu().numpy(), oracle.nhd_to_hnd(vc))
    assert np.array_equal(pools["hnd"][2].cpu().numpy(), ks, equal_nan=True)
    assert torch.equal(outs["hnd"], outs["nhd"])
    assert_attention_close(out_to_f64(outs["hnd"]), oracle_int8(case, (kc, vc, ks, vs)),
                           "INT8 HND decode_store")
