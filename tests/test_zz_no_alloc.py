"""kvc_decode_noalloc: decode for callers that cannot allocate device memory.

Some users of this library receive only their input and output buffers -- an operator
inside an inference engine that planned all of its device memory at start-up, or a serving
loop that may not call cudaMalloc (which can synchronise the whole device) while it runs.
They cannot pass kvc_decode a workspace, so kvc_decode_noalloc keeps the split partials in a
fixed scratch array inside the library instead.  These tests call it through the C ABI and
check it against kvc_decode and against the fp64 oracle, twice in a row (the scratch keeps
the previous call's data), and check that a plan too large for the scratch is refused with
a clear error.  Each test builds its own inputs, so the file passes alone in a fresh process
as well as after the other tests; it is named to be collected last, so that a run stopping
at its first failure has run every other test before it.
"""
import numpy as np
import pytest
import torch

import pagedattention_kvc_store_gb300 as kvc
from harness import MAX_ABS, MEAN_ABS, GpuRun, OracleRun, assert_attention_close, out_to_f64
from workloads import config_case

pytestmark = pytest.mark.gpu


def _decode_both(case, num_splits):
    """The same batch through kvc_decode (own workspace) and kvc_decode_noalloc."""
    g = GpuRun(case, decode=True)
    g.store()
    ref = g.attend(torch.float32, num_splits)            # kvc_decode with a workspace
    got = torch.full_like(ref, float("nan"))
    kvc.kvc_decode_noalloc(got, g.d.q, g.d.k_pool, g.d.v_pool, g.d.block_table,
                           g.d.context_lens, case.max_ctx, num_splits=num_splits)
    torch.cuda.synchronize()
    return out_to_f64(ref), out_to_f64(got)


def test_matches_decode_on_two_calls_in_a_row():
    first = config_case(2)                          # 64 sequences, 2 automatic splits
    second = config_case(2, num_seqs=40, seed=99)   # another batch, then 5 splits
    for case, splits in ((first, 0), (second, 5)):
        pool = kvc.pool_desc(torch.empty(1, case.page_size, case.kv_heads, case.head_dim))
        n, _, ws = kvc.kvc_decode_plan(case.num_seqs, case.q_heads, pool, case.max_ctx, splits)
        assert n > 1 and 0 < ws <= kvc.NOALLOC_SCRATCH_BYTES   # the scratch is really used
        ref, got = _decode_both(case, splits)
        assert np.isfinite(got).all()
        err = np.abs(got - ref)
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS
        exact, _ = OracleRun(case).attention()
        assert_attention_close(got, exact, f"kvc_decode_noalloc, {splits} splits")


def test_plan_beyond_the_scratch_is_refused():
    case = config_case(1)
    g = GpuRun(case, decode=True)
    out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, dtype=torch.bfloat16,
                      device="cuda")
    # 2048 splits of 64 positions: 16 rows x 2048 x 64 dims x 4 bytes of partials (+ lse)
    # come to just over 8 MiB, more than the scratch holds; nothing may be launched.
    with pytest.raises(kvc.KvcError) as info:
        kvc.kvc_decode_noalloc(out, g.d.q, g.d.k_pool, g.d.v_pool, g.d.block_table,
                               g.d.context_lens, 131072, num_splits=2048)
    assert info.value.status == 3 and "scratch" in str(info.value)
