"""Failure detection on the GPU without a fault: a bounded wait that nothing satisfies gives
up after about a second, the kernel records it in the device error word and returns, and the
context keeps working (the next calls run and match the oracle)."""
import time

import pytest
import torch

import pagedattention_kvc_store_gb300 as kvc
from harness import GpuRun, OracleRun, assert_attention_close, out_to_f64
from workloads import config_case

pytestmark = pytest.mark.gpu

SELFTEST_BIT = 1 << 12


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    torch.cuda.synchronize()
    kvc.kvc_device_errors()                       # clear whatever earlier tests left
    t0 = time.perf_counter()
    kvc.kvc_selftest_wait()
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    flags = kvc.kvc_device_errors()
    assert flags & SELFTEST_BIT, f"the wait did not report giving up (flags {flags:#x})"
    assert 0.2 < waited < 20.0, f"the bounded wait took {waited:.2f} s"
    assert kvc.kvc_device_errors() == 0           # reading clears the word

    case = config_case(1)
    g = GpuRun(case, decode=True)
    g.store()
    out = g.attend(torch.float32, 2)
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
    ref, _ = OracleRun(case).attention()
    assert_attention_close(out_to_f64(out), ref, "decode after the self-test")


def test_caller_error_words_stay_separate_across_streams():
    """kvc_set_error_word: two callers, each with a device word of its own, on two streams at
    once.  The self-test's give-up bit lands only in the first word, a context longer than its
    block-table row (clamped and flagged, bit 7) only in the second, the library's own words
    see neither, and with the word unset again the bits go back to kvc_device_errors."""
    torch.cuda.synchronize()
    kvc.kvc_device_errors()
    case = config_case(1)
    g = GpuRun(case, decode=True)
    g.store()
    torch.cuda.synchronize()
    over = g.d.context_lens.clone()
    over[2] = case.block_table.shape[1] * case.page_size + 5   # past its row
    word_a = torch.zeros(1, dtype=torch.int32, device="cuda")
    word_b = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, device="cuda")
    try:
        kvc.kvc_set_error_word(word_a)
        kvc.kvc_selftest_wait(sa)                            # about a second on stream a
        kvc.kvc_set_error_word(word_b)
        with torch.cuda.stream(sb):                          # meanwhile on stream b
            kvc.kvc_decode(out, g.d.q, g.d.k_pool, g.d.v_pool, g.d.block_table, over,
                           case.max_ctx, num_splits=1)
        sb.synchronize()
        assert int(word_b.item()) == 1 << 7 and int(word_a.item()) in (0, SELFTEST_BIT)
        sa.synchronize()
        assert int(word_a.item()) == SELFTEST_BIT
        assert int(word_b.item()) == 1 << 7
        assert kvc.kvc_device_errors() == 0                  # the library's words saw nothing
        # a clean call with a caller word leaves it as it was
        word_b.zero_()
        out2 = g.attend(torch.float32, 2)
        torch.cuda.synchronize()
        assert int(word_b.item()) == 0
    finally:
        kvc.kvc_set_error_word(None)
    ref, _ = OracleRun(case).attention()
    assert_attention_close(out_to_f64(out2), ref, "decode with a caller error word")
    kvc.kvc_selftest_wait()
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == SELFTEST_BIT
