"""Device group detection (kvc_shared_prefix_groups) against the oracle's groups, bit for bit,
and end to end: the groups it finds drive kvc_decode_shared_prefix to the oracle's attention."""
import numpy as np
import pytest
import torch

import pagedattention_kvc_store_gb300 as kvc
from harness import GpuRun, OracleRun, assert_attention_close, out_to_f64
from oracle.plan import groups_from_block_tables
from workloads import config_case
from workloads.device import i32_tensor

pytestmark = pytest.mark.gpu


def detect(bt: np.ndarray, ctx: np.ndarray, P: int, max_members: int):
    S = len(ctx)
    cap = S // 2
    indptr = torch.full((cap + 1,), -7, dtype=torch.int32, device="cuda")
    seqs = torch.full((max(S, 1),), -7, dtype=torch.int32, device="cuda")
    prefix = torch.full((max(cap, 1),), -7, dtype=torch.int32, device="cuda")
    n = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    kvc.kvc_shared_prefix_groups(indptr, seqs, prefix, n,
                                 i32_tensor(bt.reshape(max(S, 1), -1), "cuda"),
                                 i32_tensor(ctx, "cuda"), P, max_members)
    torch.cuda.synchronize()
    return (indptr.cpu().numpy(), seqs.cpu().numpy(), prefix.cpu().numpy(), int(n.item()))


def check_against_oracle(bt, ctx, P, max_members):
    indptr, seqs, prefix, n = detect(bt, ctx, P, max_members)
    r_indptr, r_seqs, r_prefix = groups_from_block_tables(bt.tolist(), ctx.tolist(), P,
                                                          max_members)
    assert n == len(r_prefix)
    assert indptr[: n + 1].tolist() == r_indptr
    total = r_indptr[-1]
    assert seqs[:total].tolist() == r_seqs
    assert prefix[:n].tolist() == r_prefix
    cap = len(ctx) // 2
    assert (indptr[n: cap + 1] == total).all(), "unused slots must be empty groups"
    assert (prefix[n:cap] == 0).all()
    return n


def random_tables(rng, S, W, P):
    """Runs of rows that copy a leading part of the previous row, then diverge."""
    bt = np.zeros((S, W), np.int32)
    nxt = 0
    for s in range(S):
        if s > 0 and rng.random() < 0.7:
            keep = int(rng.integers(0, W + 1))
            bt[s, :keep] = bt[s - 1, :keep]
        else:
            keep = 0
        bt[s, keep:] = np.arange(nxt, nxt + W - keep)
        nxt += W - keep
    ctx = rng.integers(0, W * P + 1, size=S).astype(np.int32)
    ctx[rng.random(S) < 0.05] = 0
    return bt, ctx


@pytest.mark.parametrize("S,W,P,mm", [(1, 4, 16, 8), (2, 4, 16, 2), (37, 9, 16, 3),
                                      (1500, 20, 32, 8), (3000, 7, 64, 64), (2049, 40, 16, 16)])
def test_random_tables_match_oracle(S, W, P, mm):
    rng = np.random.default_rng(S + W + P + mm)
    bt, ctx = random_tables(rng, S, W, P)
    check_against_oracle(bt, ctx, P, mm)


def test_long_runs_cross_tiles():
    """One run over 2,500 sequences (crossing the kernel's 1,024-sequence tiles), cut into
    chunks of 7; agreements vary along the run."""
    rng = np.random.default_rng(5)
    S, W, P = 2500, 30, 16
    bt = np.tile(np.arange(W, dtype=np.int32), (S, 1))
    cut = rng.integers(1, W, size=S)
    for s in range(S):
        bt[s, cut[s]:] = 100000 + s * W + np.arange(W - cut[s])
    ctx = np.full(S, W * P, np.int32)
    n = check_against_oracle(bt, ctx, P, 7)
    assert n == -(-S // 7) - (1 if S % 7 == 1 else 0)


def test_workload_groups_and_decode():
    """The shared-prefix workload: the device finds its 32 groups of 8 (2,048 shared
    positions), and the decode driven by them -- with every capacity slot, the unused ones
    empty -- matches the oracle."""
    case = config_case(3)
    indptr, seqs, prefix, n = detect(case.block_table, case.context_lens, case.page_size, 16)
    assert n == 32 and (prefix[:32] == 2048).all()
    g = GpuRun(case, decode=True)
    g.store()
    cap = case.num_seqs // 2
    pool = kvc.pool_desc(g.d.k_pool)
    ws = kvc.kvc_decode_shared_prefix_plan(case.num_seqs, case.q_heads, pool, case.max_ctx, cap,
                                           case.max_ctx)
    work = torch.empty(ws, dtype=torch.uint8, device="cuda")
    out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, dtype=torch.float32,
                      device="cuda")
    kvc.kvc_decode_shared_prefix(out, g.d.q, g.d.k_pool, g.d.v_pool, g.d.block_table,
                                 g.d.context_lens, case.max_ctx, i32_tensor(indptr, "cuda"),
                                 i32_tensor(seqs, "cuda"), i32_tensor(prefix, "cuda"), 16,
                                 case.max_ctx, work)
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
    ref, _ = OracleRun(case).attention()
    assert_attention_close(out_to_f64(out), ref, "decode over device-found groups")


def test_refuses_bad_arguments():
    t = torch.zeros(4, dtype=torch.int32, device="cuda")
    bt = torch.zeros(4, 2, dtype=torch.int32, device="cuda")
    for mm in (1, 65):
        with pytest.raises(kvc.KvcError) as info:
            kvc.kvc_shared_prefix_groups(t, t, t, t, bt, t, 16, mm)
        assert info.value.status == 1
