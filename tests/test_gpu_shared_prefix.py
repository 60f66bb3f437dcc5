"""GPU parity of shared-prefix (grouped) decode: groups of sequences whose block tables begin
with the same pages are decoded with the shared pages read once per group; the result must
equal the oracle's per-sequence attention and kvc_decode's."""
import numpy as np
import pytest
import torch

import pagedattention_kvc_store_gb300 as kvc
from harness import GpuRun, OracleRun, assert_attention_close, out_to_f64
from workloads import build_case, config_case
from workloads.device import i32_tensor

pytestmark = pytest.mark.gpu


def _group_arrays(case):
    groups = case.groups
    sp = case.shared_positions
    prefix = [int(sp[i]) if np.ndim(sp) else int(sp) for i in range(len(groups))]
    indptr = np.concatenate([[0], np.cumsum([len(g) for g in groups])]).astype(np.int32)
    seqs = np.concatenate([np.asarray(g, np.int32) for g in groups]) if groups else \
        np.zeros(0, np.int32)
    return indptr, seqs, np.asarray(prefix, np.int32)


def _run_shared(case, g, arrays=None):
    indptr, seqs, prefix = _group_arrays(case) if arrays is None else arrays
    max_group = max((len(x) for x in case.groups), default=1)
    max_prefix = int(prefix.max()) if prefix.size else 0
    pool = kvc.pool_desc(g.d.k_pool)
    ws = kvc.kvc_decode_shared_prefix_plan(case.num_seqs, case.q_heads, pool, case.max_ctx,
                                           len(prefix), max_prefix)
    # every byte 0xFF: a partial slot the grid failed to write (or to mark empty) reads as NaN
    work = torch.full((ws,), 0xFF, dtype=torch.uint8, device="cuda")
    out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, dtype=torch.float32,
                      device="cuda")
    kvc.kvc_decode_shared_prefix(out, g.d.q, g.d.k_pool, g.d.v_pool, g.d.block_table,
                                 g.d.context_lens, case.max_ctx, i32_tensor(indptr, "cuda"),
                                 i32_tensor(seqs, "cuda"), i32_tensor(prefix, "cuda"),
                                 max_group, max_prefix, work)
    return out_to_f64(out)


def test_shared_prefix_workload_full_size():
    case = config_case(3)
    g = GpuRun(case, decode=True)
    g.store()
    got = _run_shared(case, g)
    ref, _ = OracleRun(case).attention()
    assert_attention_close(got, ref, "shared-prefix decode (grouped)")
    plain = out_to_f64(g.attend(torch.float32, 0))
    assert np.abs(got - plain).max() < 2e-3


def _random_groups(P, max_members):
    def make(rng, ctx):
        S = len(ctx)
        order = rng.permutation(S)
        groups, prefix, k = [], [], 0
        while k < S:
            n = int(rng.integers(1, max_members + 1))
            members = [int(x) for x in order[k: k + n]]
            k += n
            if rng.random() < 0.15:
                continue                      # these sequences share nothing
            lim = (min(int(ctx[m]) for m in members) - 1) // P * P
            pre = int(rng.integers(0, lim // P + 1)) * P if lim > 0 else 0
            groups.append(members)
            prefix.append(pre)
        return dict(groups=groups, shared_positions=prefix)
    return make


@pytest.mark.parametrize("P,Hq,Hkv,D,members", [(16, 32, 8, 128, 8), (32, 16, 8, 128, 4),
                                                (64, 16, 2, 64, 8), (16, 8, 8, 64, 16),
                                                (16, 64, 8, 128, 8)])
def test_random_groups(P, Hq, Hkv, D, members):
    case = build_case(P * 3 + Hq + members, name="groups", page_size=P, q_heads=Hq,
                      kv_heads=Hkv, head_dim=D,
                      context_lens=lambda rng: rng.integers(1, 900, size=29),
                      q_lens=np.ones_like, share_groups=_random_groups(P, members))
    g = GpuRun(case, decode=True)
    g.store()
    got = _run_shared(case, g)
    ref, _ = OracleRun(case).attention()
    assert_attention_close(got, ref, f"groups {P},{Hq},{Hkv},{D},{members}")


def test_more_work_items_than_one_wave_with_empty_slots():
    """Groups x kv heads well above the prefix CTAs of one resident wave (2 per SM), so CTAs
    take several items in turn, with empty group slots between and after the real ones (the
    shape of a device-found list) and groups whose prefix is empty."""
    P, Hkv = 16, 8
    case = build_case(71, name="groups", page_size=P, q_heads=32, kv_heads=Hkv, head_dim=128,
                      context_lens=lambda rng: rng.integers(1, 260, size=240),
                      q_lens=np.ones_like, share_groups=_random_groups(P, 3))
    indptr, seqs, prefix = _group_arrays(case)
    sizes = np.diff(indptr)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert len(sizes) * Hkv > 2 * n_sm, "the case must exceed one wave of prefix CTAs"
    # an empty slot after every third group and a tail of them, as a fixed-capacity list has
    new_sizes, new_prefix = [], []
    for i, (n, pre) in enumerate(zip(sizes, prefix)):
        new_sizes.append(int(n))
        new_prefix.append(int(pre))
        if i % 3 == 2:
            new_sizes.append(0)
            new_prefix.append(0)
    new_sizes += [0] * 40
    new_prefix += [0] * 40
    arrays = (np.concatenate([[0], np.cumsum(new_sizes)]).astype(np.int32), seqs,
              np.asarray(new_prefix, np.int32))
    g = GpuRun(case, decode=True)
    g.store()
    got = _run_shared(case, g, arrays)
    ref, _ = OracleRun(case).attention()
    assert_attention_close(got, ref, "groups over several prefix items per CTA")


def test_rejects_groups_with_too_many_rows():
    case = config_case(1)
    g = GpuRun(case, decode=True)
    work = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    out = torch.empty(4, 4, 64, dtype=torch.bfloat16, device="cuda")
    one = i32_tensor(np.array([0, 4]), "cuda")
    with pytest.raises(kvc.KvcError) as info:
        kvc.kvc_decode_shared_prefix(out, g.d.q, g.d.k_pool, g.d.v_pool, g.d.block_table,
                                     g.d.context_lens, 100, one, i32_tensor(np.arange(4), "cuda"),
                                     i32_tensor(np.array([16]), "cuda"), 33, 16, work)
    assert info.value.status == 2


def test_no_device_errors_were_raised():
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_no_groups_runs_suffix_only(out_dtype):
    """No groups at all: the grid holds only suffix CTAs, each from position 0, and the result
    is the oracle's plain attention."""
    case = build_case(77, name="no-groups", page_size=16, q_heads=32, kv_heads=8, head_dim=128,
                      context_lens=lambda rng: rng.integers(1, 700, size=19),
                      q_lens=np.ones_like)
    g = GpuRun(case, decode=True)
    g.store()
    pool = kvc.pool_desc(g.d.k_pool)
    ws = kvc.kvc_decode_shared_prefix_plan(case.num_seqs, case.q_heads, pool, case.max_ctx, 0, 0)
    work = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, dtype=out_dtype,
                      device="cuda")
    none = i32_tensor(np.zeros(1, np.int32), "cuda")
    kvc.kvc_decode_shared_prefix(out, g.d.q, g.d.k_pool, g.d.v_pool, g.d.block_table,
                                 g.d.context_lens, case.max_ctx, none, none,
                                 i32_tensor(np.zeros(1, np.int32), "cuda")[:0], 1, 0, work)
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
    ref, _ = OracleRun(case).attention()
    assert_attention_close(out_to_f64(out), ref, "shared-prefix call without groups")


def test_shared_pages_and_private_copies_agree():
    """Sharing is storage: tables whose members point at one copy of the prefix pages and
    tables where every member of four groups has its own copy of them give bit-identical
    kvc_decode output; the grouped decode over the shared tables agrees with both."""
    case = config_case(3)
    g1 = GpuRun(case, decode=True)
    g1.store()
    shared_out = g1.attend(torch.float32, 0)
    grouped = _run_shared(case, g1)

    case2 = config_case(3)
    pages = case2.k_pool.shape[0]
    n_sh = case2.shared_positions // case2.page_size
    members = [m for grp in case2.groups[:4] for m in grp]
    src = np.concatenate([case2.block_table[m, :n_sh] for m in members])
    fresh = np.arange(pages, pages + len(src), dtype=np.int32)
    case2.k_pool = np.concatenate([case2.k_pool, case2.k_pool[src]])
    case2.v_pool = np.concatenate([case2.v_pool, case2.v_pool[src]])
    for i, m in enumerate(members):
        case2.block_table[m, :n_sh] = fresh[i * n_sh:(i + 1) * n_sh]
    g2 = GpuRun(case2, decode=True)
    g2.store()
    private_out = g2.attend(torch.float32, 0)
    torch.cuda.synchronize()
    assert torch.equal(private_out, shared_out)
    assert np.abs(grouped - out_to_f64(private_out)).max() < 2e-3
