"""Pins of the oracle's INT8 cache (TileInfer.jl "KV cache", section "INT8 cache"): the
quantiser against hand-worked vectors and its defining properties, the INT8 store, and
attention over INT8 pages reduced to cases the bf16 attention or a closed form fixes."""
import numpy as np
import pytest

from conftest import golden_lines
from oracle import oracle
from workloads import bf16_bits, f32_from_bf16, normal_bf16


def test_quantize_worked_vectors():
    for line in golden_lines("int8_quantize.txt"):
        vals, m, codes = line.split(" | ")
        x = bf16_bits(np.array([float(v) for v in vals.split()], dtype=np.float32))
        got_codes, scale = oracle.quantize_vector(x)
        assert scale == np.float32(np.float32(float(m)) / np.float32(127.0))
        assert got_codes.tolist() == [int(c) for c in codes.split()]


def test_quantize_properties():
    rng = np.random.default_rng(3)
    ss = np.random.SeedSequence(31)
    for i in range(200):
        x = normal_bf16(ss.spawn(1)[0], (128,))
        if i % 7 == 0:
            x = bf16_bits(f32_from_bf16(x) * np.float32(rng.choice([1e-3, 1e3])))
        codes, scale = oracle.quantize_vector(x)
        xf = f32_from_bf16(x).astype(np.float64)
        m = np.abs(xf).max()
        assert scale == np.float32(np.float32(m) / np.float32(127.0))
        assert np.abs(codes).max() == 127                         # the largest maps to +-127
        assert codes[np.argmax(np.abs(xf))] == np.sign(xf[np.argmax(np.abs(xf))]) * 127
        # reconstruction within half a step (plus fp32 rounding of the quotient)
        assert np.all(np.abs(xf - scale * codes) <= 0.5 * scale * (1 + 1e-5) + 1e-30)
        # symmetric: -x gives -codes and the same scale
        neg_codes, neg_scale = oracle.quantize_vector(x ^ np.uint16(0x8000))
        assert neg_scale == scale and np.array_equal(neg_codes, -codes)


def test_int8_vector_bytes():
    # 132 bytes per vector at head_dim 128 against 256 in bf16 (the same section's figure)
    codes, scale = oracle.quantize_vector(normal_bf16(np.random.SeedSequence(1), (128,)))
    assert codes.nbytes + np.float32(scale).nbytes == 132


def _int8_pools(pages, P, H, D):
    return (np.zeros((pages, P, H, D), np.int8), np.zeros((pages, P, H, D), np.int8),
            np.full((pages, H, P), np.nan, np.float32), np.full((pages, H, P), np.nan, np.float32))


def test_store_int8_writes_only_mapped_slots():
    pages, P, H, D = 6, 16, 2, 64
    kc, vc, ks, vs = _int8_pools(pages, P, H, D)
    ss = np.random.SeedSequence(9)
    k_new, v_new = normal_bf16(ss.spawn(1)[0], (3, H, D)), normal_bf16(ss.spawn(1)[0], (3, H, D))
    slots = np.array([17, -1, 95])
    oracle.store_int8(kc, vc, ks, vs, k_new, v_new, slots)
    for t, slot in ((0, 17), (2, 95)):
        page, off = divmod(slot, P)
        for g in range(H):
            c, s = oracle.quantize_vector(k_new[t, g])
            assert np.array_equal(kc[page, off, g], c) and ks[page, g, off] == s
            c, s = oracle.quantize_vector(v_new[t, g])
            assert np.array_equal(vc[page, off, g], c) and vs[page, g, off] == s
    written = np.zeros((pages, H, P), bool)
    written[1, :, 1] = written[5, :, 15] = True
    assert np.isnan(ks[~written]).all() and np.isnan(vs[~written]).all()
    assert np.count_nonzero(kc.reshape(pages * P, H, D).any(axis=(1, 2))) <= 2


def test_attention_int8_with_unit_scales_is_bf16_attention():
    """Scales of 1: every vector is its integer codes, exact in bf16, so attention over the
    INT8 pages must equal the bf16 attention over those integers."""
    pages, P, Hkv, Hq, D = 8, 16, 2, 8, 64
    rng = np.random.default_rng(4)
    kc = rng.integers(-127, 128, size=(pages, P, Hkv, D)).astype(np.int8)
    vc = rng.integers(-127, 128, size=(pages, P, Hkv, D)).astype(np.int8)
    ones = np.ones((pages, Hkv, P), np.float32)
    bt = rng.permutation(pages).astype(np.int32).reshape(2, 4)
    ctx = np.array([50, 37], np.int32)
    q = normal_bf16(np.random.SeedSequence(2), (2, Hq, D))
    ind = np.arange(3, dtype=np.int32)
    got, lse = oracle.attention_int8(q, kc, vc, ones, ones, bt, ctx, ind, scale=0.01)
    kb = bf16_bits(kc.astype(np.float32))
    vb = bf16_bits(vc.astype(np.float32))
    ref, ref_lse = oracle.attention(q, kb, vb, bt, ctx, ind, scale=0.01)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_attention_int8_zero_key_scales_average_values():
    """Key scales of 0 make every score 0: the output is the mean of the stored values."""
    pages, P, Hkv, Hq, D = 4, 16, 1, 2, 64
    rng = np.random.default_rng(8)
    kc = rng.integers(-127, 128, size=(pages, P, Hkv, D)).astype(np.int8)
    vc = rng.integers(-127, 128, size=(pages, P, Hkv, D)).astype(np.int8)
    ks = np.zeros((pages, Hkv, P), np.float32)
    vs = rng.uniform(0.5, 2.0, size=(pages, Hkv, P)).astype(np.float32)
    bt = np.array([[2, 0, 3]], np.int32)
    ctx = np.array([40], np.int32)
    q = normal_bf16(np.random.SeedSequence(6), (1, Hq, D))
    out, lse = oracle.attention_int8(q, kc, vc, ks, vs, bt, ctx, np.arange(2, dtype=np.int32))
    rows = [vs[bt[0, p // P], 0, p % P] * vc[bt[0, p // P], p % P, 0].astype(np.float64)
            for p in range(40)]
    np.testing.assert_allclose(out[0, 0], np.mean(rows, axis=0), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse[0], np.log(40.0), rtol=1e-12)
