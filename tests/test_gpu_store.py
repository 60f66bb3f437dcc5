"""GPU parity of slot mapping and store against the oracle: bit-exact, including every
pool entry the store must leave alone (they keep their NaN poison)."""
import numpy as np
import pytest
import torch

import pagedattention_kvc_store_gb300 as kvc
from harness import GpuRun, OracleRun, pools_bits
from workloads import build_case, config_case
from workloads.device import bf16_bits_of, bf16_tensor, i32_tensor

pytestmark = pytest.mark.gpu


def _check_store(case, decode):
    g = GpuRun(case, decode=decode)
    g.store()
    o = OracleRun(case)
    np.testing.assert_array_equal(g.slots.cpu().numpy().astype(np.int64), o.slots)
    k_bits, v_bits = pools_bits(g)
    assert np.array_equal(k_bits, o.k_pool), "K pool differs from the oracle's"
    assert np.array_equal(v_bits, o.v_pool), "V pool differs from the oracle's"


def test_tiny_decode_store_is_bit_exact():
    case = config_case(1)
    _check_store(case, decode=True)
    # the four new tokens land at offsets 0, 0, 0, 3 of their pages
    g = GpuRun(case, decode=True)
    g.store()
    assert (g.slots.cpu().numpy() % 16).tolist() == [0, 0, 0, 3]


def test_batched_decode_store_is_bit_exact():
    _check_store(config_case(2), decode=True)


@pytest.mark.parametrize("page_size", [16, 64])
def test_rewind_chunk_store_is_bit_exact(page_size):
    # 1,000 documents x 50 new tokens each: the chunk starts mid-page (offset 12 / 44)
    case = config_case(4, page_size=page_size)
    _check_store(case, decode=False)


@pytest.mark.parametrize("P", [16, 32, 64])
def test_ragged_store_random_lengths(P):
    case = build_case(100 + P, name="ragged", page_size=P, q_heads=8, kv_heads=2, head_dim=64,
                      context_lens=lambda rng: rng.integers(1, 400, size=37),
                      q_lens=lambda ctx: np.minimum(ctx, 1 + (ctx % 23)))
    _check_store(case, decode=False)


def test_negative_slots_are_skipped_and_bits_travel():
    P, H, D, pages = 16, 2, 64, 8
    rng = np.random.default_rng(5)
    pool = rng.integers(0, 2**16, size=(pages, P, H, D), dtype=np.uint16)
    k_new = rng.integers(0, 2**16, size=(5, H, D), dtype=np.uint16)
    v_new = rng.integers(0, 2**16, size=(5, H, D), dtype=np.uint16)
    k_new[0, :, :4] = [0x7FC1, 0xFF81, 0x8000, 0x0001]   # NaN payloads, -0, denormal
    slots = np.array([7, -1, 100, -5, 127], dtype=np.int32)
    kp, vp = bf16_tensor(pool, "cuda"), bf16_tensor(pool.copy(), "cuda")
    kvc.kvc_store(kp, vp, bf16_tensor(k_new, "cuda"), bf16_tensor(v_new, "cuda"),
                  i32_tensor(slots, "cuda"))
    ref_k, ref_v = pool.copy(), pool.copy()
    for t, s in enumerate(slots):
        if s >= 0:
            ref_k.reshape(-1, H, D)[s] = k_new[t]
            ref_v.reshape(-1, H, D)[s] = v_new[t]
    assert np.array_equal(bf16_bits_of(kp), ref_k)
    assert np.array_equal(bf16_bits_of(vp), ref_v)


def test_slot_mapping_negative_position_gives_minus_one():
    bt = i32_tensor(np.array([[3, 0, 5, 0]]), "cuda")
    ctx = i32_tensor(np.array([1]), "cuda")
    indptr = i32_tensor(np.array([0, 3]), "cuda")
    slots = torch.empty(3, dtype=torch.int32, device="cuda")
    kvc.kvc_slot_mapping(slots, bt, ctx, indptr, 4, max_q_len=3)
    assert slots.cpu().tolist() == [-1, -1, 12]


@pytest.mark.parametrize("decode,cfg", [(True, 2), (False, 4)])
def test_store_and_slot_mapping_read_pinned_host_inputs(decode, cfg):
    """kvc_slot_mapping's tables and kvc_store's new keys and values may sit in pinned host
    memory: the slots and the pools come out bit for bit as from device inputs (and as the
    oracle's)."""
    case = config_case(cfg, num_seqs=96) if not decode else config_case(cfg)
    g = GpuRun(case, decode=decode)
    d = g.d
    host = {n: getattr(d, n).cpu().pin_memory() for n in ("block_table", "context_lens",
                                                           "q_indptr", "k_new", "v_new")}
    kvc.kvc_slot_mapping(g.slots, host["block_table"], host["context_lens"],
                         None if decode else host["q_indptr"], case.page_size,
                         max_q_len=case.max_q_len)
    kvc.kvc_store(d.k_pool, d.v_pool, host["k_new"], host["v_new"], g.slots)
    torch.cuda.synchronize()
    assert kvc.kvc_device_errors() == 0
    o = OracleRun(case)
    np.testing.assert_array_equal(g.slots.cpu().numpy().astype(np.int64), o.slots)
    k_bits, v_bits = pools_bits(g)
    assert np.array_equal(k_bits, o.k_pool)
    assert np.array_equal(v_bits, o.v_pool)


def test_store_refuses_pageable_host_inputs():
    from pagedattention_kvc_store_gb300.kvc import lib, pool_desc, _ptr
    case = config_case(1)
    g = GpuRun(case, decode=True)
    d = g.d
    kvc.kvc_slot_mapping(g.slots, d.block_table, d.context_lens, None, case.page_size)
    host_k = np.zeros(d.k_new.numel() + 16, dtype=np.uint16)
    addr = (host_k.ctypes.data + 15) // 16 * 16
    import ctypes
    st = lib().kvc_store(_ptr(d.k_pool), _ptr(d.v_pool), pool_desc(d.k_pool),
                         ctypes.c_void_p(addr), _ptr(d.v_new), _ptr(g.slots),
                         int(g.slots.shape[0]), None)
    assert st == 1 and b"pinned host" in lib().kvc_last_error()
