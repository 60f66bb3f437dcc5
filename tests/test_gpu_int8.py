"""INT8 pages on the GPU against the oracle (TileInfer.jl "KV cache", section "INT8 cache").

The cached positions of a seeded bf16 case are quantised into INT8 pages by the oracle; every
slot that holds no position keeps random codes and a NaN scale (so a masked position that
leaked into a sum would show).  The new tokens are then quantised and stored by
kvc_store_int8 (codes and scales bit-exact against the oracle's store) and kvc_decode_int8
attends over the pages (within the attention tolerance of the oracle's fp64 attention over
scale * code)."""
import numpy as np
import pytest
import torch

import pagedattention_kvc_store_gb300 as kvc
from harness import assert_attention_close, int8_pages, out_to_f64, sample_seqs
from oracle import oracle
from workloads import build_case, config_case
from workloads.device import bf16_tensor, i32_tensor

pytestmark = pytest.mark.gpu


def run_int8(case, num_splits=0, out_dtype=torch.float32):
    kc, vc, ks, vs = int8_pages(case)
    dev = dict(kc=torch.from_numpy(kc).cuda(), vc=torch.from_numpy(vc).cuda(),
               ks=torch.from_numpy(ks).cuda(), vs=torch.from_numpy(vs).cuda())
    bt, ctx = i32_tensor(case.block_table, "cuda"), i32_tensor(case.context_lens, "cuda")
    slots = torch.empty(case.num_tokens, dtype=torch.int32, device="cuda")
    kvc.kvc_slot_mapping(slots, bt, ctx, None, case.page_size)
    kvc.kvc_store_int8(dev["kc"], dev["vc"], dev["ks"], dev["vs"],
                       bf16_tensor(case.k_new, "cuda"), bf16_tensor(case.v_new, "cuda"), slots)
    oracle.store_int8(kc, vc, ks, vs, case.k_new, case.v_new,
                      slots.cpu().numpy().astype(np.int64))
    assert np.array_equal(dev["kc"].cpu().numpy(), kc), "K codes differ from the oracle's"
    assert np.array_equal(dev["vc"].cpu().numpy(), vc), "V codes differ from the oracle's"
    for name, ref in (("ks", ks), ("vs", vs)):
        got = dev[name].cpu().numpy()
        assert np.array_equal(np.isnan(got), np.isnan(ref)), f"{name}: NaN pattern"
        assert np.array_equal(got[~np.isnan(ref)], ref[~np.isnan(ref)]), f"{name} differs"
    out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, dtype=out_dtype,
                      device="cuda")
    pool = kvc.int8_pool_desc(dev["kc"])
    _, _, ws = kvc.kvc_decode_int8_plan(case.num_seqs, case.q_heads, pool, case.max_ctx,
                                        num_splits)
    work = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    kvc.kvc_decode_int8(out, bf16_tensor(case.q, "cuda"), dev["kc"], dev["vc"], dev["ks"],
                        dev["vs"], bt, ctx, case.max_ctx, num_splits=num_splits, workspace=work)
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
    return out, (kc, vc, ks, vs)


def oracle_int8(case, pools, seqs=None):
    kc, vc, ks, vs = pools
    if seqs is None:
        seqs = np.arange(case.num_seqs)
    ind = np.arange(len(seqs) + 1, dtype=np.int32)
    ref, _ = oracle.attention_int8(case.q[seqs], kc, vc, ks, vs, case.block_table[seqs],
                                   case.context_lens[seqs], ind, num_threads=16)
    return ref


@pytest.mark.parametrize("P", [16, 32, 64])
@pytest.mark.parametrize("G", [1, 4, 8])
def test_int8_decode_ragged(P, G):
    case = build_case(700 + P + G, name="int8", page_size=P, q_heads=2 * G, kv_heads=2,
                      head_dim=128, context_lens=lambda rng: rng.integers(1, 700, size=24),
                      q_lens=lambda ctx: np.ones_like(ctx))
    for splits in (1, 3, 0):
        out, pools = run_int8(case, num_splits=splits)
        assert_attention_close(out_to_f64(out), oracle_int8(case, pools),
                               f"INT8 decode P={P} G={G} splits={splits}")


def test_int8_decode_batched_workload():
    """The batched-decode workload (64 sequences, ctx U[512, 4096], 32/8 heads, D 128, P 16)
    on INT8 pages, bf16 output, checked on sampled sequences."""
    case = config_case(2)
    out, pools = run_int8(case, out_dtype=torch.bfloat16)
    seqs = sample_seqs(case.num_seqs, 12)
    assert_attention_close(out_to_f64(out)[seqs], oracle_int8(case, pools, seqs),
                           "INT8 batched decode")


def test_int8_decode_batched_workload_f32_every_sequence():
    """The same workload with fp32 output: all 64 sequences, held to the plain attention
    tolerance (no allowance for output rounding)."""
    case = config_case(2)
    out, pools = run_int8(case, out_dtype=torch.float32)
    assert_attention_close(out_to_f64(out), oracle_int8(case, pools),
                           "INT8 batched decode, fp32 output, every sequence")


@pytest.mark.parametrize("P", [16, 32, 64])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_int8_decode_head_dim_64(P, G):
    """head_dim 64 (64-byte code rows, 64-byte swizzle): the store's codes and scales bit-exact
    and the decode within tolerance, split and whole, fp32 and bf16 output."""
    case = build_case(720 + P + G, name="int8-d64", page_size=P, q_heads=2 * G, kv_heads=2,
                      head_dim=64, context_lens=lambda rng: rng.integers(1, 700, size=20),
                      q_lens=lambda ctx: np.ones_like(ctx))
    for splits in (1, 3, 0):
        out, pools = run_int8(case, num_splits=splits)
        assert_attention_close(out_to_f64(out), oracle_int8(case, pools),
                               f"INT8 decode D=64 P={P} G={G} splits={splits}")
    # bf16 output: the attention tolerance plus the output's own rounding (half an ulp),
    # since scale * code is seldom a bf16 number
    out, pools = run_int8(case, out_dtype=torch.bfloat16)
    ref = oracle_int8(case, pools)
    err = np.abs(out_to_f64(out) - ref)
    assert (err - 2.0 ** -8 * np.abs(ref)).max() <= 1e-2 and err.mean() <= 1e-3


def test_int8_tiny_decode_head_dim_64():
    """The tiny workload (head_dim 64, contexts 1, 17, 33, 100) on INT8 pages, every sequence."""
    case = config_case(1)
    out, pools = run_int8(case, num_splits=2)
    assert_attention_close(out_to_f64(out), oracle_int8(case, pools), "INT8 tiny decode")


def test_int8_single_position_is_its_stored_vector():
    case = build_case(77, name="one", page_size=16, q_heads=4, kv_heads=2, head_dim=128,
                      context_lens=lambda rng: np.array([1, 1, 2]),
                      q_lens=lambda ctx: np.ones_like(ctx))
    out, (kc, vc, ks, vs) = run_int8(case)
    for s in (0, 1):
        slot = oracle.slot_of_position(case.block_table, s, 0, 16)
        page, off = divmod(slot, 16)
        for h in range(case.q_heads):
            g = h // 2
            want = vs[page, g, off] * vc[page, off, g].astype(np.float64)
            # the probability 1 times the value scale enters the PV product as bf16
            np.testing.assert_allclose(out_to_f64(out)[s, h], want, rtol=2.0 ** -8, atol=1e-6)


def decode_int8_only(case, pools, ctx, num_splits):
    """kvc_decode_int8 over given pools with the given context lengths (fp32 output)."""
    kc, vc, ks, vs = (torch.from_numpy(a).cuda() for a in pools)
    bt, ctx_t = i32_tensor(case.block_table, "cuda"), i32_tensor(ctx, "cuda")
    out = torch.full((case.num_seqs, case.q_heads, case.head_dim), float("nan"),
                     device="cuda")
    pool = kvc.int8_pool_desc(kc)
    _, _, ws = kvc.kvc_decode_int8_plan(case.num_seqs, case.q_heads, pool, case.max_ctx,
                                        num_splits)
    work = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    kvc.kvc_decode_int8(out, bf16_tensor(case.q, "cuda"), kc, vc, ks, vs, bt, ctx_t,
                        case.max_ctx, num_splits=num_splits, workspace=work)
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
    return out_to_f64(out)


@pytest.mark.parametrize("splits", [0, 1, 2, 7])
def test_int8_partition_across_sequences(splits):
    """The positions of all sequences are cut into equal runs per kv head: runs that cross
    sequence boundaries, sequences much longer than a run (their rows merged from many
    pieces), contexts of 1 .. 127 positions, and sequences with no positions between them
    (their rows are 0)."""
    ctx = np.array([1, 5000, 3, 1, 64, 65, 9000, 2, 127, 1, 3000, 17])
    case = build_case(1300, name="int8-partition", page_size=16, q_heads=8, kv_heads=2,
                      head_dim=128, context_lens=lambda rng: ctx,
                      q_lens=lambda c: np.ones_like(c))
    out, pools = run_int8(case, num_splits=splits)
    assert_attention_close(out_to_f64(out), oracle_int8(case, pools),
                           f"INT8 partition splits={splits}")
    ctx0 = ctx.copy()
    ctx0[[0, 3, 9]] = 0
    got = decode_int8_only(case, pools, ctx0, splits)
    assert not got[[0, 3, 9]].any(), "a sequence with no positions has rows of 0"
    keep = np.flatnonzero(ctx0 > 0)
    kc, vc, ks, vs = pools
    ref, _ = oracle.attention_int8(case.q[keep], kc, vc, ks, vs, case.block_table[keep],
                                   ctx0[keep], np.arange(len(keep) + 1, dtype=np.int32),
                                   num_threads=16)
    assert_attention_close(got[keep], ref, f"INT8 partition with empty sequences {splits}")


def test_int8_more_ctas_than_blocks():
    """Fewer 64-position blocks than planned runs: only as many runs as blocks are used."""
    case = build_case(1301, name="int8-few-blocks", page_size=16, q_heads=8, kv_heads=2,
                      head_dim=128, context_lens=lambda rng: np.array([1, 2, 70]),
                      q_lens=lambda c: np.ones_like(c))
    for splits in (0, 9):
        out, pools = run_int8(case, num_splits=splits)
        assert_attention_close(out_to_f64(out), oracle_int8(case, pools),
                               f"INT8 few blocks splits={splits}")


@pytest.mark.parametrize("num_seqs", [256, 300])
def test_int8_large_batch_merge(num_seqs):
    """Many short sequences (each run of the cut crosses many of them, most units are whole
    and the rest are merged), with empty sequences among them, the default cut and an
    explicit one."""
    case = build_case(1302 + num_seqs, name="int8-many", page_size=16, q_heads=8, kv_heads=2,
                      head_dim=128, context_lens=lambda rng: rng.integers(1, 400, size=num_seqs),
                      q_lens=lambda c: np.ones_like(c))
    for splits in (0, 2):
        out, pools = run_int8(case, num_splits=splits)
        assert_attention_close(out_to_f64(out), oracle_int8(case, pools),
                               f"INT8 {num_seqs} sequences splits={splits}")
    ctx0 = case.context_lens.copy()
    ctx0[::7] = 0
    got = decode_int8_only(case, pools, ctx0, 0)
    assert not got[ctx0 == 0].any(), "a sequence with no positions has rows of 0"
    keep = np.flatnonzero(ctx0 > 0)
    kc, vc, ks, vs = pools
    ref, _ = oracle.attention_int8(case.q[keep], kc, vc, ks, vs, case.block_table[keep],
                                   ctx0[keep], np.arange(len(keep) + 1, dtype=np.int32),
                                   num_threads=16)
    assert_attention_close(got[keep], ref, f"INT8 {num_seqs} sequences with empty ones")
