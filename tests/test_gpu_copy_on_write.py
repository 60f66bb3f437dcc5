"""Copy-on-write on the GPU: kvc_copy_pages is bit-exact against the oracle's page copy, and
the flow of "KV Cache Management and PagedAttention", "Split shared blocks when a write is
needed" (two responses continue one common input whose last page is partly filled) gives each
response attention over its own continuation, equal to the oracle on the same tables."""
import numpy as np
import pytest
import torch

import pagedattention_kvc_store_gb300 as kvc
from harness import assert_attention_close, out_to_f64
from oracle import oracle
from workloads import BF16_NAN, PageAllocator, normal_bf16
from workloads.device import bf16_bits_of, bf16_tensor, i32_tensor

pytestmark = pytest.mark.gpu


def test_copy_pages_bit_exact():
    rng = np.random.default_rng(11)
    pages, P, H, D = 64, 16, 8, 128
    k = rng.integers(0, 1 << 16, size=(pages, P, H, D), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(pages, P, H, D), dtype=np.uint16)
    k[5, 3, 1, :4] = [0x7FC1, 0xFF81, 0x8000, 0x0001]   # NaN payloads, -0, a denormal
    perm = rng.permutation(pages)
    src, dst = perm[:20].astype(np.int32), perm[20:40].astype(np.int32)
    kd, vd = bf16_tensor(k, "cuda"), bf16_tensor(v, "cuda")
    kvc.kvc_copy_pages(kd, vd, i32_tensor(src, "cuda"), i32_tensor(dst, "cuda"))
    oracle.copy_pages(k, v, src, dst)
    assert np.array_equal(bf16_bits_of(kd), k)
    assert np.array_equal(bf16_bits_of(vd), v)
    assert kvc.kvc_device_errors() == 0


def test_copy_pages_skips_pages_outside_the_pool():
    k = np.zeros((4, 16, 2, 64), dtype=np.uint16)
    kd, vd = bf16_tensor(k, "cuda"), bf16_tensor(k.copy(), "cuda")
    kvc.kvc_copy_pages(kd, vd, i32_tensor(np.array([0, 9]), "cuda"),
                       i32_tensor(np.array([1, 2]), "cuda"))
    assert kvc.kvc_device_errors() != 0          # the out-of-pool copy was flagged ...
    assert kvc.kvc_device_errors() == 0          # ... and the word cleared on read


@pytest.mark.parametrize("common", [40, 48])     # partly filled / full last page
def test_two_responses_fork_and_write(common):
    P, Hq, Hkv, D, pages = 16, 8, 2, 64, 12
    ss = np.random.SeedSequence(4242 + common)
    a = PageAllocator(pages, P, permutation=np.random.default_rng(ss.spawn(1)[0]).permutation(pages))
    k = np.full((pages, P, Hkv, D), BF16_NAN, dtype=np.uint16)
    v = k.copy()
    # the common input: positions 0 .. common-1 of sequence 0
    a.reserve(0, common)
    kc, vc = normal_bf16(ss.spawn(1)[0], (common, Hkv, D)), normal_bf16(ss.spawn(1)[0], (common, Hkv, D))
    slots = np.array([a.pages[0][p // P] * P + p % P for p in range(common)])
    oracle.store(k, v, kc, vc, slots)
    a.fork(1, 0)
    kd, vd = bf16_tensor(k, "cuda"), bf16_tensor(v, "cuda")
    # response 1 writes a0, response 2 writes b0, at position `common`
    new_k = normal_bf16(ss.spawn(1)[0], (2, Hkv, D))
    new_v = normal_bf16(ss.spawn(1)[0], (2, Hkv, D))
    copies = a.reserve(0, 1) + a.reserve(1, 1)
    assert len(copies) == (1 if common % P else 0)
    if copies:
        src = np.array([c[0] for c in copies], dtype=np.int32)
        dst = np.array([c[1] for c in copies], dtype=np.int32)
        kvc.kvc_copy_pages(kd, vd, i32_tensor(src, "cuda"), i32_tensor(dst, "cuda"))
        oracle.copy_pages(k, v, src, dst)
    bt = a.table([0, 1], width=16)
    ctx = np.array([common + 1, common + 1], dtype=np.int32)
    btd, ctxd = i32_tensor(bt, "cuda"), i32_tensor(ctx, "cuda")
    sl = torch.empty(2, dtype=torch.int32, device="cuda")
    kvc.kvc_slot_mapping(sl, btd, ctxd, None, P)
    kvc.kvc_store(kd, vd, bf16_tensor(new_k, "cuda"), bf16_tensor(new_v, "cuda"), sl)
    oracle.store(k, v, new_k, new_v, oracle.slot_mapping(bt, ctx, np.arange(3, dtype=np.int32), P))
    # the pools match the oracle bit for bit, the two responses' last positions differ
    assert np.array_equal(bf16_bits_of(kd), k) and np.array_equal(bf16_bits_of(vd), v)
    assert bt[0, 0] == bt[1, 0]                   # page 0 still shared
    last = (common) // P
    assert bt[0, last] != bt[1, last]             # each response has its own written page
    q = normal_bf16(ss.spawn(1)[0], (2, Hq, D))
    out = torch.empty((2, Hq, D), dtype=torch.float32, device="cuda")
    pool = kvc.pool_desc(kd)
    _, _, ws = kvc.kvc_decode_plan(2, Hq, pool, common + 1, 0)
    work = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    kvc.kvc_decode(out, bf16_tensor(q, "cuda"), kd, vd, btd, ctxd, common + 1, workspace=work)
    ref, _ = oracle.attention(q, k, v, bt, ctx, np.arange(3, dtype=np.int32))
    assert_attention_close(out_to_f64(out), ref, "decode after copy-on-write")
    assert kvc.kvc_device_errors() == 0
