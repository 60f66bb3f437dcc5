"""Pins for the CPU oracle: it is checked against the pages' worked examples, against a
library attention routine on unpaged data, against closed forms and invariants -- never
against itself or the CUDA path.  CPU only."""
import math

import numpy as np
import pytest
import torch

from conftest import golden_lines
from oracle import oracle
from oracle.plan import computed_tokens, sharing_plan
from workloads import BF16_NAN, bf16_bits, f32_from_bf16

# ----------------------------------------------------------------------------------------
# Address rule and slot mapping (worked examples)
# ----------------------------------------------------------------------------------------


def _address_cases():
    for line in golden_lines("address_rule.txt"):
        P, table, pos, lblock, off, page, slot = [f.strip() for f in line.split("|")]
        yield (int(P), [int(x) for x in table.split()], int(pos), int(lblock), int(off),
               int(page), int(slot))


@pytest.mark.parametrize("case", list(_address_cases()))
def test_address_rule_worked_examples(case):
    P, table, pos, lblock, off, page, slot = case
    assert table[lblock] == page and page * P + off == slot  # the fixture is consistent
    assert oracle.slot_of_position(np.array([table]), 0, pos, P) == slot


def test_slot_mapping_worked_example_growth():
    # Sequence B grows from 7 to 9 positions: tokens at positions 7 and 8 in one step.
    bt = np.array([[3, 0, 5, 0]], dtype=np.int32)
    slots = oracle.slot_mapping(bt, np.array([9]), np.array([0, 2]), 4)
    assert slots.tolist() == [3, 20]


def test_slot_mapping_is_injective_for_private_tables():
    rng = np.random.default_rng(7)
    P, S = 16, 9
    ctx = rng.integers(1, 200, size=S)
    pages = [-(-int(c) // P) for c in ctx]
    perm = rng.permutation(sum(pages))
    bt = np.zeros((S, 16), dtype=np.int32)
    k = 0
    for s in range(S):
        bt[s, : pages[s]] = perm[k: k + pages[s]]
        k += pages[s]
    # every cached position of every sequence as a "new token"
    slots = oracle.slot_mapping(bt, ctx, np.concatenate([[0], np.cumsum(ctx)]), P)
    assert len(set(slots.tolist())) == int(ctx.sum())
    assert slots.min() >= 0 and slots.max() < sum(pages) * P


# ----------------------------------------------------------------------------------------
# Store
# ----------------------------------------------------------------------------------------


def test_store_writes_only_mapped_rows_and_keeps_bits():
    rng = np.random.default_rng(3)
    pages, P, H, D = 6, 4, 2, 8
    k_pool = rng.integers(0, 2**16, size=(pages, P, H, D), dtype=np.uint16)
    v_pool = rng.integers(0, 2**16, size=(pages, P, H, D), dtype=np.uint16)
    k0, v0 = k_pool.copy(), v_pool.copy()
    k_new = rng.integers(0, 2**16, size=(3, H, D), dtype=np.uint16)
    v_new = rng.integers(0, 2**16, size=(3, H, D), dtype=np.uint16)
    k_new[0, 0, 0] = 0x7FC1          # NaN payload must travel
    v_new[2, 1, 3] = 0x8000          # negative zero must travel
    slots = np.array([5, -1, 22], dtype=np.int64)
    oracle.store(k_pool, v_pool, k_new, v_new, slots)
    flat_k, flat_v = k_pool.reshape(-1, H, D), v_pool.reshape(-1, H, D)
    assert np.array_equal(flat_k[5], k_new[0]) and np.array_equal(flat_v[5], v_new[0])
    assert np.array_equal(flat_k[22], k_new[2]) and np.array_equal(flat_v[22], v_new[2])
    changed = np.nonzero((k_pool != k0).any(axis=(2, 3)).reshape(-1))[0].tolist()
    assert set(changed) <= {5, 22}
    other = np.ones(pages * P, dtype=bool)
    other[[5, 22]] = False
    assert np.array_equal(flat_k[other], k0.reshape(-1, H, D)[other])
    assert np.array_equal(flat_v[other], v0.reshape(-1, H, D)[other])


# ----------------------------------------------------------------------------------------
# Attention: against torch scaled_dot_product_attention on unpaged data (fp64)
# ----------------------------------------------------------------------------------------


def _rand_bf16(rng, shape):
    return bf16_bits(rng.standard_normal(shape).astype(np.float32))


def _contiguous_case(rng, ctxs, q_lens, P, Hq, Hkv, D):
    """Each sequence gets its own run of pages in order, so the pool, reshaped to
    [num_pages * P, Hkv, D], holds sequence s's positions contiguously from its first page
    on; no address arithmetic is needed to read them back."""
    pages = [-(-c // P) for c in ctxs]
    first_page = np.concatenate([[0], np.cumsum(pages)])
    n_pages = int(first_page[-1]) or 1
    bt = np.zeros((len(ctxs), max(max(pages), 1)), dtype=np.int32)
    for s, n in enumerate(pages):
        bt[s, :n] = np.arange(first_page[s], first_page[s] + n)
    k_pool = _rand_bf16(rng, (n_pages, P, Hkv, D))
    v_pool = _rand_bf16(rng, (n_pages, P, Hkv, D))
    q_indptr = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = _rand_bf16(rng, (int(q_indptr[-1]), Hq, D))
    return dict(q=q, k_pool=k_pool, v_pool=v_pool, bt=bt, ctx=np.array(ctxs, np.int32),
                q_indptr=q_indptr, first_page=first_page)


def _sdpa_reference(c, s, i, P, Hq, Hkv, scale=None):
    """torch SDPA (fp64) for new token i of sequence s: keys 0 .. position, unpaged."""
    ctx = int(c["ctx"][s])
    q_len = int(c["q_indptr"][s + 1] - c["q_indptr"][s])
    position = ctx - q_len + i
    start = int(c["first_page"][s]) * P
    to64 = lambda bits: torch.from_numpy(f32_from_bf16(bits).astype(np.float64))
    keys = to64(c["k_pool"].reshape(-1, Hkv, c["k_pool"].shape[-1])[start: start + position + 1])
    vals = to64(c["v_pool"].reshape(-1, Hkv, c["v_pool"].shape[-1])[start: start + position + 1])
    G = Hq // Hkv
    keys = keys.permute(1, 0, 2).repeat_interleave(G, dim=0)      # [Hq, n_keys, D]
    vals = vals.permute(1, 0, 2).repeat_interleave(G, dim=0)
    qv = to64(c["q"][int(c["q_indptr"][s]) + i])[:, None, :]       # [Hq, 1, D]
    kw = {} if scale is None else dict(scale=scale)
    out = torch.nn.functional.scaled_dot_product_attention(qv, keys, vals, **kw)
    return out[:, 0, :].numpy()


@pytest.mark.parametrize("P,Hq,Hkv,D", [(16, 4, 2, 64), (4, 8, 2, 16), (16, 8, 8, 32),
                                        (64, 8, 1, 128)])
def test_decode_matches_sdpa_on_unpaged_data(P, Hq, Hkv, D):
    rng = np.random.default_rng(P * 1000 + Hq * 10 + D)
    ctxs = [1, 5, P, P + 1, 3 * P - 1, 100]
    c = _contiguous_case(rng, ctxs, [1] * len(ctxs), P, Hq, Hkv, D)
    out, _ = oracle.attention(c["q"], c["k_pool"], c["v_pool"], c["bt"], c["ctx"],
                              c["q_indptr"])
    for s in range(len(ctxs)):
        ref = _sdpa_reference(c, s, 0, P, Hq, Hkv)
        np.testing.assert_allclose(out[s], ref, rtol=0, atol=1e-12)


def test_custom_scale_matches_sdpa():
    rng = np.random.default_rng(11)
    c = _contiguous_case(rng, [37], [1], 16, 4, 2, 32)
    out, _ = oracle.attention(c["q"], c["k_pool"], c["v_pool"], c["bt"], c["ctx"],
                              c["q_indptr"], scale=0.3)
    np.testing.assert_allclose(out[0], _sdpa_reference(c, 0, 0, 16, 4, 2, scale=0.3),
                               rtol=0, atol=1e-12)


@pytest.mark.parametrize("prefix,q_len", [(0, 7), (13, 5), (300, 50), (16, 16)])
def test_append_matches_sdpa_per_query(prefix, q_len):
    # new token i sits at position prefix + i and sees keys 0 .. prefix + i
    rng = np.random.default_rng(prefix * 100 + q_len)
    P, Hq, Hkv, D = 16, 8, 2, 32
    c = _contiguous_case(rng, [prefix + q_len], [q_len], P, Hq, Hkv, D)
    out, _ = oracle.attention(c["q"], c["k_pool"], c["v_pool"], c["bt"], c["ctx"],
                              c["q_indptr"])
    for i in range(q_len):
        np.testing.assert_allclose(out[i], _sdpa_reference(c, 0, i, P, Hq, Hkv),
                                   rtol=0, atol=1e-12)


def test_append_without_prefix_is_causal_self_attention():
    rng = np.random.default_rng(5)
    P, Hq, Hkv, D, n = 16, 4, 4, 16, 21
    c = _contiguous_case(rng, [n], [n], P, Hq, Hkv, D)
    out, _ = oracle.attention(c["q"], c["k_pool"], c["v_pool"], c["bt"], c["ctx"],
                              c["q_indptr"])
    to64 = lambda b: torch.from_numpy(f32_from_bf16(b).astype(np.float64))
    qq = to64(c["q"]).permute(1, 0, 2)
    kk = to64(c["k_pool"].reshape(-1, Hkv, D)[:n]).permute(1, 0, 2)
    vv = to64(c["v_pool"].reshape(-1, Hkv, D)[:n]).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, is_causal=True)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------------------
# Attention: invariants and closed forms
# ----------------------------------------------------------------------------------------


def _scattered_case(rng, ctxs, q_lens, P, Hq, Hkv, D, spare=3):
    pages = [-(-c // P) for c in ctxs]
    n_pages = sum(pages) + spare
    perm = rng.permutation(n_pages)
    bt = np.zeros((len(ctxs), max(pages) + 2), dtype=np.int32)
    k = 0
    for s, n in enumerate(pages):
        bt[s, :n] = perm[k: k + n]
        k += n
    k_pool = _rand_bf16(rng, (n_pages, P, Hkv, D))
    v_pool = _rand_bf16(rng, (n_pages, P, Hkv, D))
    q_indptr = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = _rand_bf16(rng, (int(q_indptr[-1]), Hq, D))
    return q, k_pool, v_pool, bt, np.array(ctxs, np.int32), q_indptr


def test_physical_placement_does_not_change_the_result():
    # Moving pages to other physical places must leave attention unchanged ("KV Cache
    # Management and PagedAttention", "Compute attention over scattered KV").
    rng = np.random.default_rng(21)
    q, kp, vp, bt, ctx, ind = _scattered_case(rng, [1, 17, 40, 64, 99], [1, 1, 3, 1, 9],
                                              16, 8, 2, 32)
    out1, lse1 = oracle.attention(q, kp, vp, bt, ctx, ind)
    relabel = rng.permutation(kp.shape[0])           # page i moves to relabel[i]
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[relabel], vp2[relabel] = kp, vp
    bt2 = relabel[bt].astype(np.int32)
    out2, lse2 = oracle.attention(q, kp2, vp2, bt2, ctx, ind)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def test_unused_slots_and_foreign_pages_are_excluded():
    # "KV Cache Management and PagedAttention", "Compute attention over scattered KV": B at
    # position 8 uses 9 positions (4 in P3, 4 in P0, 1 in P5); C's pages P1, P4 and the
    # three unused slots of P5 take no part.  Poison them with NaN.
    rng = np.random.default_rng(8)
    P, Hkv, D, Hq = 4, 1, 8, 2
    kp = _rand_bf16(rng, (6, P, Hkv, D))
    vp = _rand_bf16(rng, (6, P, Hkv, D))
    bt = np.array([[3, 0, 5, 0]], dtype=np.int32)
    q = _rand_bf16(rng, (1, Hq, D))
    ref, _ = oracle.attention(q, kp, vp, bt, np.array([9]), np.array([0, 1]))
    kp2, vp2 = kp.copy(), vp.copy()
    for pool in (kp2, vp2):
        pool[1] = BF16_NAN
        pool[4] = BF16_NAN
        pool[2] = BF16_NAN
        pool[5, 1:] = BF16_NAN
    out, _ = oracle.attention(q, kp2, vp2, bt, np.array([9]), np.array([0, 1]))
    assert np.isfinite(out).all() and np.array_equal(out, ref)


def test_single_position_returns_its_value_exactly():
    rng = np.random.default_rng(1)
    q, kp, vp, bt, ctx, ind = _scattered_case(rng, [1], [1], 16, 4, 2, 64)
    out, lse = oracle.attention(q, kp, vp, bt, ctx, ind)
    slot_v = vp[bt[0, 0], 0].astype(np.uint16)       # position 0 = offset 0 of page bt[0,0]
    slot_k = kp[bt[0, 0], 0]
    for h in range(4):
        g = h // 2
        np.testing.assert_array_equal(out[0, h], f32_from_bf16(slot_v[g]).astype(np.float64))
        x = float(np.dot(f32_from_bf16(q[0, h]).astype(np.float64),
                         f32_from_bf16(slot_k[g]).astype(np.float64))) / 8.0
        assert lse[0, h] == pytest.approx(x, abs=1e-12)


def test_equal_keys_or_zero_query_average_the_values():
    rng = np.random.default_rng(2)
    c = _contiguous_case(rng, [37], [1], 16, 4, 2, 16)
    kp_eq = c["k_pool"].copy()
    kp_eq[...] = c["k_pool"][0, 0, 0][None, None, None, :]     # every key identical
    out, lse = oracle.attention(c["q"], kp_eq, c["v_pool"], c["bt"], c["ctx"], c["q_indptr"])
    vals = f32_from_bf16(c["v_pool"].reshape(-1, 2, 16)[:37]).astype(np.float64)
    mean_v = vals.mean(axis=0)                                 # [Hkv, D]
    for h in range(4):
        np.testing.assert_allclose(out[0, h], mean_v[h // 2], rtol=0, atol=1e-12)
        x = float(f32_from_bf16(c["q"][0, h]).astype(np.float64)
                  @ f32_from_bf16(c["k_pool"][0, 0, 0]).astype(np.float64)) / 4.0
        assert lse[0, h] == pytest.approx(x + math.log(37), abs=1e-12)
    q0 = np.zeros_like(c["q"])
    out0, lse0 = oracle.attention(q0, c["k_pool"], c["v_pool"], c["bt"], c["ctx"],
                                  c["q_indptr"])
    for h in range(4):
        np.testing.assert_allclose(out0[0, h], mean_v[h // 2], rtol=0, atol=1e-12)
        assert lse0[0, h] == pytest.approx(math.log(37), abs=1e-12)


def test_two_positions_closed_form():
    # softmax over two scores x0, x1 is v0 + (v1 - v0) * sigmoid(x1 - x0)
    P, Hkv, D = 4, 1, 2
    kp = np.full((2, P, Hkv, D), BF16_NAN, dtype=np.uint16)
    vp = np.full((2, P, Hkv, D), BF16_NAN, dtype=np.uint16)
    kp[1, 0, 0] = bf16_bits(np.array([0.5, -1.0]))
    kp[1, 1, 0] = bf16_bits(np.array([2.0, 0.25]))
    vp[1, 0, 0] = bf16_bits(np.array([1.0, -3.0]))
    vp[1, 1, 0] = bf16_bits(np.array([-2.0, 4.0]))
    q = bf16_bits(np.array([[[1.5, 2.0]]]))
    out, lse = oracle.attention(q, kp, vp, np.array([[1]]), np.array([2]), np.array([0, 1]))
    x0 = (1.5 * 0.5 + 2.0 * -1.0) / math.sqrt(2)
    x1 = (1.5 * 2.0 + 2.0 * 0.25) / math.sqrt(2)
    sig = 1.0 / (1.0 + math.exp(-(x1 - x0)))
    expect = np.array([1.0 + (-2.0 - 1.0) * sig, -3.0 + (4.0 + 3.0) * sig])
    np.testing.assert_allclose(out[0, 0], expect, rtol=0, atol=1e-14)
    assert lse[0, 0] == pytest.approx(max(x0, x1) + math.log1p(math.exp(-abs(x1 - x0))),
                                      abs=1e-14)


def test_empty_context_gives_zero_and_minus_infinity():
    rng = np.random.default_rng(4)
    q, kp, vp, bt, ctx, ind = _scattered_case(rng, [5], [1], 4, 2, 1, 8)
    out, lse = oracle.attention(q, kp, vp, bt, np.array([0]), ind)
    assert (out == 0).all() and np.isneginf(lse).all()


# ----------------------------------------------------------------------------------------
# Split partials and their log-sum-exp merge
# ----------------------------------------------------------------------------------------


@pytest.mark.parametrize("chunk", [1, 16, 48, 1000])
def test_split_partials_merge_to_the_whole(chunk):
    rng = np.random.default_rng(chunk)
    ctxs = [1, 33, 100, 150]
    q, kp, vp, bt, ctx, ind = _scattered_case(rng, ctxs, [1] * 4, 16, 8, 2, 32)
    full, full_lse = oracle.attention(q, kp, vp, bt, ctx, ind)
    n_split = -(-max(ctxs) // chunk)
    po = np.zeros((4, 8, n_split, 32))
    pl = np.zeros((4, 8, n_split))
    for j in range(n_split):
        lo = np.full(4, j * chunk, np.int32)
        hi = np.full(4, (j + 1) * chunk, np.int32)
        o, l = oracle.attention(q, kp, vp, bt, ctx, ind, key_lo=lo, key_hi=hi)
        po[:, :, j], pl[:, :, j] = o, l
    merged, merged_lse = oracle.merge(po.reshape(32, n_split, 32), pl.reshape(32, n_split))
    np.testing.assert_allclose(merged.reshape(4, 8, 32), full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(merged_lse.reshape(4, 8), full_lse, rtol=0, atol=1e-12)


def test_merge_of_one_split_is_identity_and_empty_splits_are_ignored():
    rng = np.random.default_rng(9)
    o = rng.standard_normal((3, 1, 16))
    l = rng.standard_normal((3, 1))
    m, ml = oracle.merge(o, l)
    np.testing.assert_allclose(m, o[:, 0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(ml, l[:, 0], rtol=0, atol=1e-15)
    o2 = np.concatenate([o, np.full((3, 2, 16), np.nan)], axis=1)
    l2 = np.concatenate([l, np.full((3, 2), -np.inf)], axis=1)
    m2, ml2 = oracle.merge(o2, l2)
    np.testing.assert_allclose(m2, m, rtol=0, atol=1e-15)
    assert np.array_equal(ml2, ml)
    m3, ml3 = oracle.merge(np.zeros((2, 4, 16)), np.full((2, 4), -np.inf))
    assert (m3 == 0).all() and np.isneginf(ml3).all()


# ----------------------------------------------------------------------------------------
# Append consistency
# ----------------------------------------------------------------------------------------


def test_append_of_one_token_is_decode_and_chunks_compose():
    rng = np.random.default_rng(12)
    P, Hq, Hkv, D = 16, 8, 2, 32
    q, kp, vp, bt, ctx, _ = _scattered_case(rng, [200], [100], P, Hq, Hkv, D)
    whole, _ = oracle.attention(q, kp, vp, bt, ctx, np.array([0, 100]))
    # the last token alone, as decode
    last, _ = oracle.attention(q[99:], kp, vp, bt, ctx, np.array([0, 1]))
    assert np.array_equal(last[0], whole[99])
    # first chunk of 50 at context 150, then the next 50 at context 200
    a, _ = oracle.attention(q[:50], kp, vp, bt, np.array([150]), np.array([0, 50]))
    b, _ = oracle.attention(q[50:], kp, vp, bt, np.array([200]), np.array([0, 50]))
    assert np.array_equal(np.concatenate([a, b]), whole)


def test_thread_count_does_not_change_the_result():
    rng = np.random.default_rng(13)
    q, kp, vp, bt, ctx, ind = _scattered_case(rng, [9, 70, 33, 1, 128], [1, 5, 2, 1, 7],
                                              16, 8, 4, 32)
    a, la = oracle.attention(q, kp, vp, bt, ctx, ind, num_threads=1)
    b, lb = oracle.attention(q, kp, vp, bt, ctx, ind, num_threads=3)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


# ----------------------------------------------------------------------------------------
# Sharing plan
# ----------------------------------------------------------------------------------------


def test_sharing_plan_worked_example():
    g = {ln.split()[0]: ln.split()[1:] for ln in golden_lines("sharing_plan.txt")}
    P = int(g["page_size"][0])
    lengths = [int(x) for x in g["lengths"]]
    trace = np.random.default_rng(0).integers(0, 50000, size=max(lengths))
    docs = [trace[:n] for n in lengths]
    order, parent, shared = sharing_plan(docs, P)
    assert order == [int(x) for x in g["order"]]
    assert parent == [None if x == "None" else int(x) for x in g["parent"]]
    assert shared == [int(x) for x in g["shared"]]
    assert computed_tokens(docs, shared) == int(g["computed"][0])
    assert sum(lengths) == int(g["unshared"][0])


def test_sharing_plan_follows_parent_links_and_caps_the_last_token():
    P = 16
    base = list(range(100, 164))                  # 64 common tokens
    docs = [base + [1, 2, 3], base + [5, 6], base + [7], base[:32], base[:33]]
    order, parent, shared = sharing_plan(docs, P)
    # sorted: base[:32] < base[:33] < base+[1..] < base+[5..] < base+[7]
    assert order == [3, 4, 0, 1, 2]
    assert shared[3] == 0 and parent[3] is None
    assert shared[4] == 32 and parent[4] == 3      # lcp 32, len-1 = 32 -> 32
    # doc 0: lcp 33 -> 32.  Its predecessor, doc 4, reuses all 32 itself, so the plan
    # follows doc 4's parent link to doc 3, which supplies those pages.
    assert shared[0] == 32 and parent[0] == 3
    assert shared[1] == 64 and parent[1] == 0      # lcp 64; predecessor doc 0 shares 32 < 64
    assert shared[2] == 64 and parent[2] == 0      # lcp 64 with doc 1 which reuses all 64


def test_sharing_plan_last_token_cap():
    P = 16
    docs = [list(range(32)), list(range(32))]      # identical: cap at len - 1 = 31 -> 16
    order, parent, shared = sharing_plan(docs, P)
    assert shared == [0, 16] and parent == [None, 0]


def test_slot_mapping_marks_tokens_without_a_position_as_padding():
    bt = np.array([[3, 0, 5, 0]], dtype=np.int32)
    slots = oracle.slot_mapping(bt, np.array([1]), np.array([0, 3]), 4)
    assert slots.tolist() == [-1, -1, 12]


def test_hnd_layout_address_rule():
    """HND pools (TileInfer.jl's (head_dim, page_size, kv_heads, num_pages) column-major array):
    the worked addresses of tests/golden/hnd_layout.txt, and the oracle's layout conversion
    puts every value at its NHD address."""
    P, H, D, pages = 4, 2, 3, 3
    hnd = np.arange(pages * H * P * D, dtype=np.uint16).reshape(pages, H, P, D)
    nhd = oracle.hnd_to_nhd(hnd)
    for line in golden_lines("hnd_layout.txt"):
        p, h, o, d, flat_hnd, flat_nhd = (int(v) for v in line.split(" | "))
        assert hnd.reshape(-1)[flat_hnd] == hnd[p, h, o, d]
        assert nhd.reshape(-1)[flat_nhd] == hnd[p, h, o, d]
    assert np.array_equal(oracle.nhd_to_hnd(nhd), hnd)


def test_hnd_store_and_attention_match_nhd():
    """The same logical cache in either layout: the store writes the same values and
    attention gives bit-identical fp64 results."""
    from workloads import build_case

    case = build_case(51, name="hnd", page_size=16, q_heads=8, kv_heads=2, head_dim=64,
                      context_lens=lambda rng: rng.integers(1, 90, size=6),
                      q_lens=lambda ctx: np.minimum(ctx, 3))
    slots = oracle.slot_mapping(case.block_table, case.context_lens, case.q_indptr,
                                case.page_size)
    k_n, v_n = case.k_pool.copy(), case.v_pool.copy()
    oracle.store(k_n, v_n, case.k_new, case.v_new, slots)
    k_h, v_h = oracle.nhd_to_hnd(case.k_pool), oracle.nhd_to_hnd(case.v_pool)
    oracle.store(k_h, v_h, case.k_new, case.v_new, slots, layout="hnd")
    assert np.array_equal(oracle.hnd_to_nhd(k_h), k_n)
    assert np.array_equal(oracle.hnd_to_nhd(v_h), v_n)
    a_n = oracle.attention(case.q, k_n, v_n, case.block_table, case.context_lens, case.q_indptr)
    a_h = oracle.attention(case.q, k_h, v_h, case.block_table, case.context_lens, case.q_indptr,
                           layout="hnd")
    assert np.array_equal(a_n[0], a_h[0]) and np.array_equal(a_n[1], a_h[1], equal_nan=True)
