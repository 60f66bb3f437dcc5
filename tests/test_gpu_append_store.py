"""Fused store + append (kvc_append_store) on the GPU.

kvc_append_store must leave the pools exactly as kvc_store with kvc_slot_mapping's slots
leaves them (bit-exact against the oracle's store, including every slot it must not touch),
and return kvc_append's output: within the attention tolerance of the oracle, and bit for bit
what the separate slot mapping + store + append calls give (the same operands meet in the same
order; only where they come from differs)."""
import numpy as np
import pytest
import torch

import pagedattention_kvc_store_gb300 as kvc
from harness import GpuRun, OracleRun, assert_attention_close, out_to_f64, sample_seqs
from oracle import oracle
from workloads import build_case, config_case
from workloads.device import bf16_bits_of, bf16_tensor, to_device

pytestmark = pytest.mark.gpu


def fused(case, out_dtype=torch.float32, layout="nhd"):
    """(out, k_pool bits, v_pool bits) of kvc_append_store on a fresh copy of the case."""
    d = to_device(case)
    kp, vp = d.k_pool, d.v_pool
    if layout == "hnd":
        kp = bf16_tensor(oracle.nhd_to_hnd(case.k_pool), "cuda")
        vp = bf16_tensor(oracle.nhd_to_hnd(case.v_pool), "cuda")
    out = torch.empty(case.num_tokens, case.q_heads, case.head_dim, dtype=out_dtype,
                      device="cuda")
    kvc.kvc_append_store(out, d.q, d.k_new, d.v_new, kp, vp, d.block_table, d.q_indptr,
                         d.context_lens, case.max_q_len, case.max_ctx, layout=layout)
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
    return out, bf16_bits_of(kp), bf16_bits_of(vp)


def separate(case, out_dtype=torch.float32):
    g = GpuRun(case, decode=False)
    g.store()
    out = g.attend(out_dtype)
    torch.cuda.synchronize()
    return out, bf16_bits_of(g.d.k_pool), bf16_bits_of(g.d.v_pool)


def check(case, what, layout="nhd", seqs=None):
    o = OracleRun(case)
    out, kb, vb = fused(case, layout=layout)
    k_ref, v_ref = o.k_pool, o.v_pool
    if layout == "hnd":
        k_ref, v_ref = oracle.nhd_to_hnd(k_ref), oracle.nhd_to_hnd(v_ref)
    assert np.array_equal(kb, k_ref), f"{what}: K pool differs from the oracle's store"
    assert np.array_equal(vb, v_ref), f"{what}: V pool differs from the oracle's store"
    if seqs is None:
        ref, _ = o.attention()
        assert_attention_close(out_to_f64(out), ref, what)
    else:
        ref, _, rows = o.attention(seqs)
        assert_attention_close(out_to_f64(out)[rows], ref, what)
    return out


@pytest.mark.parametrize("P,Hq,Hkv,D", [(16, 32, 8, 128), (32, 8, 8, 64), (64, 16, 2, 128),
                                        (16, 16, 2, 64), (64, 8, 1, 128)])
def test_append_store_ragged(P, Hq, Hkv, D):
    """Ragged contexts and chunks: chunks that start inside a page and on a page boundary,
    span several pages and 128-position blocks, and (q_len * G > 256) several tile pairs."""
    case = build_case(P + Hq * 5 + D, name="append-store", page_size=P, q_heads=Hq,
                      kv_heads=Hkv, head_dim=D,
                      context_lens=lambda rng: rng.integers(1, 600, size=23),
                      q_lens=lambda ctx: np.minimum(ctx, 1 + (ctx * 7) % 173))
    out = check(case, f"append_store {P},{Hq},{Hkv},{D}")
    ref_out, _, _ = separate(case)
    assert torch.equal(out, ref_out), "fused and separate store + append differ"


def test_append_store_edges():
    """No prefix (ctx == q_len), a chunk inside one page, chunks ending exactly at a page or
    block end, q_len = 1, and a long chunk of many tile pairs (each stores its own pages)."""
    ctx = np.array([1, 2, 17, 64, 65, 128, 129, 256, 300, 5, 640, 1000, 33, 48])
    qlen = np.array([1, 2, 17, 64, 1, 128, 1, 64, 300, 5, 1, 512, 3, 32])
    case = build_case(91, name="append-store-edges", page_size=16, q_heads=8, kv_heads=2,
                      head_dim=128, context_lens=lambda rng: ctx, q_lens=lambda c: qlen)
    out = check(case, "append_store edges")
    ref_out, _, _ = separate(case)
    assert torch.equal(out, ref_out)


@pytest.mark.parametrize("P", [16, 64])
def test_append_store_rewind_workload(P):
    """The rewind-append workload (1,000 documents, 300 cached + 50 new, 32 / 8 heads): pools
    bit-exact over the whole pool, output checked on sampled documents and equal to the
    separate calls'."""
    case = config_case(4, page_size=P)
    seqs = sample_seqs(case.num_seqs, 40, seed=P + 1)
    out = check(case, f"append_store rewind P={P}", seqs=seqs)
    ref_out, _, _ = separate(case)
    assert torch.equal(out, ref_out)


def test_append_store_hnd():
    case = build_case(92, name="append-store-hnd", page_size=32, q_heads=16, kv_heads=4,
                      head_dim=128, context_lens=lambda rng: rng.integers(1, 500, size=17),
                      q_lens=lambda ctx: np.minimum(ctx, 1 + (ctx * 5) % 97))
    check(case, "append_store HND", layout="hnd")


def test_append_store_bf16_output_and_graph_replay():
    """bf16 output, and a captured graph replayed twice: the second replay re-stores the same
    rows, so pools and output are unchanged."""
    case = build_case(93, name="append-store-graph", page_size=16, q_heads=8, kv_heads=2,
                      head_dim=128, context_lens=lambda rng: rng.integers(40, 400, size=12),
                      q_lens=lambda ctx: np.full_like(ctx, 37))
    d = to_device(case)
    out = torch.empty(case.num_tokens, case.q_heads, case.head_dim, dtype=torch.bfloat16,
                      device="cuda")
    s = torch.cuda.Stream()

    def call():
        kvc.kvc_append_store(out, d.q, d.k_new, d.v_new, d.k_pool, d.v_pool, d.block_table,
                             d.q_indptr, d.context_lens, case.max_q_len, case.max_ctx)
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    first = out.clone()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, first)
    o = OracleRun(case)
    assert np.array_equal(bf16_bits_of(d.k_pool), o.k_pool)
    assert np.array_equal(bf16_bits_of(d.v_pool), o.v_pool)
    ref, _ = o.attention()
    assert_attention_close(out_to_f64(out), ref, "append_store bf16 output")


@pytest.mark.parametrize("P", [16, 64])
def test_append_store_context_past_the_row(P):
    """A context longer than its block-table row (a caller error): kvc_append_store must leave
    the pools exactly as kvc_slot_mapping + kvc_store do -- the chunk's tokens the row covers
    at their own slots, the rest skipped -- and both paths flag bit 1 << 7.  Sequence 0 fills
    its 16-entry row exactly (ctx = 16 P); on the device its context is then raised by 10, so
    the chunk's last 10 tokens fall past the row and the others land on its own pages.  At
    P = 64 the call stores the whole chunk first, at P = 16 the append writes the later pages."""
    cap = 16 * P
    ctx = np.array([cap, 200, 75, 211, 40])
    qlen = np.array([50, 50, 9, 120, 40])
    case = build_case(94 + P, name="append-store-over", page_size=P, q_heads=16, kv_heads=4,
                      head_dim=128, context_lens=lambda rng: ctx, q_lens=lambda c: qlen,
                      bt_width=16)
    assert case.block_table.shape[1] * P == cap
    over = case.context_lens.copy()
    over[0] += 10

    def run(fused_call):
        d = to_device(case)
        d.context_lens.copy_(torch.from_numpy(over.astype(np.int32)))
        out = torch.zeros(case.num_tokens, case.q_heads, case.head_dim, dtype=torch.float32,
                          device="cuda")
        kvc.kvc_device_errors()
        if fused_call:
            kvc.kvc_append_store(out, d.q, d.k_new, d.v_new, d.k_pool, d.v_pool, d.block_table,
                                 d.q_indptr, d.context_lens, case.max_q_len, cap)
        else:
            slots = torch.empty(case.num_tokens, dtype=torch.int32, device="cuda")
            kvc.kvc_slot_mapping(slots, d.block_table, d.context_lens, d.q_indptr, P,
                                 max_q_len=case.max_q_len)
            kvc.kvc_store(d.k_pool, d.v_pool, d.k_new, d.v_new, slots)
            kvc.kvc_append(out, d.q, d.k_pool, d.v_pool, d.block_table, d.q_indptr,
                           d.context_lens, case.max_q_len, cap)
        torch.cuda.synchronize()
        flags = kvc.kvc_device_errors()
        return out, bf16_bits_of(d.k_pool), bf16_bits_of(d.v_pool), flags

    out_f, kf, vf, flags_f = run(True)
    out_s, ks, vs, flags_s = run(False)
    assert flags_f & (1 << 7) and flags_s & (1 << 7)
    assert np.array_equal(kf, ks), "K pools differ from slot mapping + store"
    assert np.array_equal(vf, vs), "V pools differ from slot mapping + store"
    # the chunk's first 40 tokens of sequence 0 were stored (at positions cap - 40 .. cap - 1),
    # its last 10 were not
    pos = np.arange(cap - 40, cap)
    slots0 = case.block_table[0][pos // P].astype(np.int64) * P + pos % P
    flat_k = kf.reshape(-1, case.kv_heads, case.head_dim)
    assert np.array_equal(flat_k[slots0], case.k_new[:40])
    # the other sequences' outputs are untouched by sequence 0's error
    rows = slice(int(case.q_indptr[1]), case.num_tokens)
    assert torch.equal(out_f[rows], out_s[rows])


def test_append_store_page_outside_the_pool():
    """A block-table entry past the pool (a caller error) on a page that holds only chunk
    tokens: kvc_append_store must leave the pools exactly as kvc_slot_mapping + kvc_store do
    (that page's tokens skipped, every other one stored) and both paths flag bit 1 << 6.
    Sequence 0 has 200 positions, 50 of them new (positions 150 .. 199): its entry 10 (positions
    160 .. 175) is set to the pool's page count on the device.  In the fused call the append
    reads the chunk from k_new and writes its later pages itself; the separate append reads
    that page through the pool's tensor map, past its end (zeros), so sequence 0's output
    differs between the two and only the others are compared."""
    P = 16
    ctx = np.array([200, 211, 75, 90, 40])
    qlen = np.array([50, 50, 9, 33, 40])
    case = build_case(96, name="append-store-page-out", page_size=P, q_heads=16, kv_heads=4,
                      head_dim=128, context_lens=lambda rng: ctx, q_lens=lambda c: qlen)
    num_pages = case.k_pool.shape[0]
    bad_table = case.block_table.copy()
    bad_table[0, 10] = num_pages

    def run(fused_call):
        d = to_device(case)
        d.block_table.copy_(torch.from_numpy(bad_table.astype(np.int32)))
        out = torch.zeros(case.num_tokens, case.q_heads, case.head_dim, dtype=torch.float32,
                          device="cuda")
        kvc.kvc_device_errors()
        if fused_call:
            kvc.kvc_append_store(out, d.q, d.k_new, d.v_new, d.k_pool, d.v_pool, d.block_table,
                                 d.q_indptr, d.context_lens, case.max_q_len, case.max_ctx)
        else:
            slots = torch.empty(case.num_tokens, dtype=torch.int32, device="cuda")
            kvc.kvc_slot_mapping(slots, d.block_table, d.context_lens, d.q_indptr, P,
                                 max_q_len=case.max_q_len)
            kvc.kvc_store(d.k_pool, d.v_pool, d.k_new, d.v_new, slots)
            kvc.kvc_append(out, d.q, d.k_pool, d.v_pool, d.block_table, d.q_indptr,
                           d.context_lens, case.max_q_len, case.max_ctx)
        torch.cuda.synchronize()
        flags = kvc.kvc_device_errors()
        return out, bf16_bits_of(d.k_pool), bf16_bits_of(d.v_pool), flags

    out_f, kf, vf, flags_f = run(True)
    out_s, ks, vs, flags_s = run(False)
    assert flags_f & (1 << 6) and flags_s & (1 << 6)
    assert np.array_equal(kf, ks), "K pools differ from slot mapping + store"
    assert np.array_equal(vf, vs), "V pools differ from slot mapping + store"
    # sequence 0's chunk tokens on its other new pages were stored
    pos = np.arange(176, 200)
    slots0 = case.block_table[0][pos // P].astype(np.int64) * P + pos % P
    flat_k = kf.reshape(-1, case.kv_heads, case.head_dim)
    assert np.array_equal(flat_k[slots0], case.k_new[26:50])
    rows = slice(int(case.q_indptr[1]), case.num_tokens)
    assert torch.equal(out_f[rows], out_s[rows])
