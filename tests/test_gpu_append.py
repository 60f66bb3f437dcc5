"""GPU parity of paged append (causal chunked prefill over a cached prefix) against the
fp64 oracle, including the KV-rewind flow: append, truncate, append again over stale slots."""
import numpy as np
import pytest
import torch

import pagedattention_kvc_store_gb300 as kvc
from harness import GpuRun, OracleRun, assert_attention_close, out_to_f64
from workloads import bf16_bits, build_case, config_case, f32_from_bf16, normal_bf16
from workloads.device import bf16_tensor, i32_tensor

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("page_size", [16, 64])
def test_rewind_append_full_size(page_size):
    """The rewind workload at full size (1,000 documents x 50 new tokens over 300 cached, 32 /
    8 heads), every document against the oracle."""
    case = config_case(4, page_size=page_size)
    g = GpuRun(case, decode=False)
    g.store()
    out = out_to_f64(g.attend(torch.bfloat16))
    ref, _ = OracleRun(case).attention()
    assert_attention_close(out, ref, f"rewind append P={page_size}")


def test_two_chunks_compose_to_one():
    """Appending 50 tokens and then 50 more over the cached first 50 gives, row for row, what
    one append of all 100 gives (the same keys and causal limits; different tiles, so within
    fp32 rounding)."""
    n, P, Hq, Hkv, D = 12, 16, 32, 8, 128
    case = build_case(4321, name="compose", page_size=P, q_heads=Hq, kv_heads=Hkv, head_dim=D,
                      context_lens=lambda rng: np.full(n, 100), q_lens=lambda c: np.full(n, 100))
    g = GpuRun(case, decode=False)
    g.store()                              # all 100 tokens of every document are now cached
    d = g.d
    whole = torch.empty(n * 100, Hq, D, dtype=torch.float32, device="cuda")
    kvc.kvc_append(whole, d.q, d.k_pool, d.v_pool, d.block_table, d.q_indptr, d.context_lens,
                   100, 100)
    q = d.q.view(n, 100, Hq, D)
    halves = []
    for lo, ctx in ((0, 50), (50, 100)):
        part = torch.empty(n * 50, Hq, D, dtype=torch.float32, device="cuda")
        kvc.kvc_append(part, q[:, lo:lo + 50].contiguous().view(n * 50, Hq, D), d.k_pool,
                       d.v_pool, d.block_table, i32_tensor(np.arange(0, n * 50 + 1, 50), "cuda"),
                       i32_tensor(np.full(n, ctx), "cuda"), 50, ctx)
        halves.append(part.view(n, 50, Hq, D))
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
    two = torch.cat(halves, dim=1).view(n * 100, Hq, D)
    assert (two - whole).abs().max().item() < 2e-3
    ref, _ = OracleRun(case).attention()
    assert_attention_close(out_to_f64(whole), ref, "append of 100")


@pytest.mark.parametrize("P,Hq,Hkv,D", [(16, 32, 8, 128), (32, 8, 8, 64), (64, 16, 2, 128),
                                        (16, 16, 2, 64), (64, 8, 1, 128)])
def test_append_ragged_shapes(P, Hq, Hkv, D):
    case = build_case(P + Hq * 3 + D, name="ragged-append", page_size=P, q_heads=Hq,
                      kv_heads=Hkv, head_dim=D,
                      context_lens=lambda rng: rng.integers(1, 420, size=23),
                      q_lens=lambda ctx: np.minimum(ctx, 1 + (ctx * 7) % 97))
    g = GpuRun(case, decode=False)
    g.store()
    for dtype in (torch.float32, torch.bfloat16):
        out = out_to_f64(g.attend(dtype))
        ref, _ = OracleRun(case).attention()
        assert_attention_close(out, ref, f"ragged append {P},{Hq},{Hkv},{D},{dtype}")


def test_append_without_prefix_and_single_token():
    # ctx == q_len: plain causal self-attention; q_len == 1: decode
    ctx = np.array([1, 2, 17, 64, 65, 130, 5, 300])
    qlen = np.array([1, 2, 17, 64, 1, 1, 5, 1])
    case = build_case(77, name="edges", page_size=16, q_heads=8, kv_heads=2, head_dim=128,
                      context_lens=lambda rng: ctx, q_lens=lambda c: qlen)
    g = GpuRun(case, decode=False)
    g.store()
    out = out_to_f64(g.attend(torch.float32))
    ref, _ = OracleRun(case).attention()
    assert_attention_close(out, ref, "append edges")


def test_append_of_one_token_matches_decode():
    case = config_case(2, num_seqs=24)
    g = GpuRun(case, decode=False)       # same case through the append path
    g.store()
    out_a = out_to_f64(g.attend(torch.float32))
    gd = GpuRun(case, decode=True)
    gd.store()
    out_d = out_to_f64(gd.attend(torch.float32, 1))
    assert np.abs(out_a - out_d).max() < 2e-3


def test_kv_rewind_truncate_and_second_question():
    # Quail "KV", "KV rewind": keep the document's KV, drop the question's, ask the next one.
    n_docs = 64
    case = config_case(4, page_size=16, num_seqs=n_docs)
    g = GpuRun(case, decode=False)
    g.store()
    first = out_to_f64(g.attend(torch.bfloat16))
    o = OracleRun(case)
    ref1, _ = o.attention()
    assert_attention_close(first, ref1, "first question")

    # truncate every document back to its 300 cached positions: pages 22 -> 19
    alloc = case.allocator
    for s in case.seqs:
        alloc.truncate(s, 300)
        assert len(alloc.pages[s]) == 19
    # the second question: 50 new tokens per document, pages reserved again
    for s in case.seqs:
        alloc.reserve(s, 50)
    case.block_table = alloc.table(case.seqs, case.block_table.shape[1])
    ss = np.random.SeedSequence(4242).spawn(2)
    case.q = normal_bf16(ss[0], case.q.shape)
    new = normal_bf16(ss[1], (2,) + case.k_new.shape)
    case.k_new, case.v_new = np.ascontiguousarray(new[0]), np.ascontiguousarray(new[1])

    # GPU: continue on the same device pools (stale slots 300.. still hold question 1)
    g.d.block_table = i32_tensor(case.block_table, "cuda")
    g.d.q = bf16_tensor(case.q, "cuda")
    g.d.k_new = bf16_tensor(case.k_new, "cuda")
    g.d.v_new = bf16_tensor(case.v_new, "cuda")
    g.store()
    second = out_to_f64(g.attend(torch.bfloat16))
    # oracle: continue on its own pools after its own first store
    case.k_pool, case.v_pool = o.k_pool, o.v_pool
    ref2, _ = OracleRun(case).attention()
    assert_attention_close(second, ref2, "second question after rewind")
    assert np.abs(second - first).max() > 0.1   # a different question, a different answer


def test_append_when_later_keys_dominate():
    # Keys of later pages are scaled up so each row's running max jumps by far more than
    # 2^8 mid-stream: the kernel must rescale what it has accumulated.
    case = build_case(31, name="rising", page_size=16, q_heads=16, kv_heads=2, head_dim=128,
                      context_lens=lambda rng: rng.integers(150, 400, size=9),
                      q_lens=lambda ctx: np.minimum(ctx, 40))
    for s in case.seqs:
        for k, page in enumerate(case.allocator.pages[s]):
            f = np.float32(1.0 + 6.0 * k)          # page k holds positions 16k .. 16k+15
            vals = f32_from_bf16(case.k_pool[page]) * f
            case.k_pool[page] = np.where(case.k_pool[page] == 0x7FC0, case.k_pool[page],
                                         bf16_bits(vals))
    g = GpuRun(case, decode=False)
    g.store()
    out = out_to_f64(g.attend(torch.float32))
    ref, _ = OracleRun(case).attention()
    assert_attention_close(out, ref, "rising keys")


def test_no_device_errors_were_raised():
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
