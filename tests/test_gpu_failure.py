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
