// kvc_append_tc.cu -- causal chunked prefill over a paged cached prefix on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// What it computes: Quail "KV", "KV rewind" and "Prefix sharing"; TileInfer.jl "KV cache",
// "Prefix reuse in chat".  New token i of a sequence (ctx positions, q_len new) sits at
// position ctx - q_len + i and attends to positions 0 .. ctx - q_len + i, read in place from
// the pages its block table lists.
//
// Tiling: the rows of one (sequence, kv head) are its (new token, query head of the group)
// pairs, token-major, 128 per tile (the tcgen05 M).  One CTA per (row tile, kv head,
// sequence):
//   warp 0      TMA: the 128-row query tile once, then 64-position K/V stages (one box per
//               page and 64-column half, 128-byte swizzle) through a 2-deep ring;
//   warp 1      allocates TMEM and issues the MMAs from one thread:
//                 S = Q K^T   (M 128, N 64, K head_dim)   into TMEM columns [D, D+64)
//                 O += P V    (M 128, N head_dim, K 64)   into TMEM columns [0, D), with P
//                                                        read from TMEM (two buffers)
//               and zeroes V rows past the last visible position, so that NaN or Inf left
//               in unused slots never meets a zero probability inside the tensor core;
//   warps 2-5   softmax: thread r owns row r (TMEM lane r): reads its S row, applies the
//               scale and the causal limit, keeps a running max / sum, writes P (bf16 pairs)
//               into one of two TMEM buffers for the PV MMA -- so block b + 1's P can be
//               written while block b's PV product still reads the other -- and at the end
//               normalises its O row from TMEM through shared memory to global memory.
// The running max is updated lazily: O is rescaled (in TMEM) only when a row's max grows by
// more than 2^8, so a block's exponentials do not wait for the previous PV product.  The
// result is exact either way; probabilities are then at most 2^8 before normalisation.
#include <math.h>

#include "kvc_device.cuh"
#include "kvc_launch.h"

namespace kvc {

namespace {

__device__ uint32_t g_append_tc_errors;

constexpr int kM = 128;            // rows per tile
constexpr int kBN = kStageKeys;    // positions per stage (64)
constexpr int kStages = 2;
constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;

template <int D>
struct TcGeom {
    static constexpr int kHalves = D / 64;
    static constexpr int kQBytes = kHalves * kM * 128;
    static constexpr int kTileBytes = kHalves * kBN * 128;   // K or V of one stage
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kOffStages = kQBytes;
    static constexpr int kOffBar = kOffStages + kStages * kStageBytes;
    static constexpr size_t kSmemBytes = kOffBar + 128;   // base is 1024-aligned
    // TMEM: O [0, D), S [D, D + 64), P buffers [D + 64, D + 96) and [D + 96, D + 128)
    static constexpr uint32_t kTmemCols = 256;
    static constexpr uint32_t kColS = D;
    static constexpr uint32_t kColP = D + kBN;
    static_assert(D + kBN + kBN <= static_cast<int>(kTmemCols), "TMEM layout");
};

struct Args {
    void *out;
    int out_f32;
    const int32_t *block_table;
    int bt_stride;
    const int32_t *q_indptr;
    const int32_t *context_lens;
    int q_heads, group, page_size;
    float scale_log2;
};

// Barrier slots after the P buffer.
enum BarIndex : int {
    kBarKvFull = 0,                 // [kStages]
    kBarKvEmpty = kBarKvFull + kStages,
    kBarQFull = kBarKvEmpty + kStages,
    kBarSFull,
    kBarSFree,
    kBarPFull,                      // [2]: one per P buffer
    kBarPvDone = kBarPFull + 2,     // [2]
    kBarDrain = kBarPvDone + 2,
    kBarCount
};

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    paged_append_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                           const __grid_constant__ CUtensorMap tmap_k,
                           const __grid_constant__ CUtensorMap tmap_v, const Args a)
{
    using Geom = TcGeom<D>;
    constexpr int kHalves = D / 64;

    // The swizzled tiles need a 1024-byte-aligned base; the dynamic shared window of a kernel
    // with no static shared memory starts there, which is checked rather than padded for (the
    // padding would cost the second CTA per SM).
    extern __shared__ __align__(1024) uint8_t smem[];
    if ((smem_addr(smem) & 1023u) != 0) {
        if (threadIdx.x == 0)
            atomicOr(&g_append_tc_errors, kErrSmemAlign);
        return;
    }
    uint8_t *sQ = smem;
    uint8_t *sStages = smem + Geom::kOffStages;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Geom::kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kBarCount);

    const int tile = blockIdx.x;
    const int kvh = blockIdx.y;
    const int s = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.group;
    const int P = a.page_size;
    const int tok0 = a.q_indptr[s];
    const int q_len = a.q_indptr[s + 1] - tok0;
    int ctx = a.context_lens[s];
    if (ctx > a.bt_stride * P) {
        if (threadIdx.x == 0 && tile == 0)
            atomicOr(&g_append_tc_errors, kErrContextRange);
        ctx = a.bt_stride * P;
    }
    const int rows = q_len * G;
    const int row_begin = tile * kM;
    if (row_begin >= rows)
        return;
    const int row_last = min(rows, row_begin + kM) - 1;
    const int n_keys = min(ctx, ctx - q_len + row_last / G + 1);
    if (n_keys <= 0)
        return;
    const int n_blocks = (n_keys + kBN - 1) / kBN;

    // Producer state (warp 0).  The query tile and the first stages are issued before the
    // CTA-wide barrier below, so the loads overlap the TMEM allocation.
    const int32_t *bt_row = a.block_table + static_cast<size_t>(s) * a.bt_stride;
    const int n_pages = (n_keys + P - 1) / P;
    int cached_base = -32;
    int cached_page = 0;
    int issued = 0;
    uint64_t policy = 0;
    // Load the K and V pages of stage b (all lanes of warp 0; lane 0 issues the copies).
    auto produce_block = [&](int b) {
        const int st = b % kStages;
        const int key0 = b * kBN;
        const int np = (min(kBN, n_keys - key0) + P - 1) / P;
        if (lane == 0)
            mbar_arrive_expect_tx(&bars[kBarKvFull + st], static_cast<uint32_t>(np * P * D * 2 * 2));
        uint8_t *kdst = sStages + st * Geom::kStageBytes;
        uint8_t *vdst = kdst + Geom::kTileBytes;
        for (int i = 0; i < np; ++i) {
            const int lp = key0 / P + i;
            if (lp >= cached_base + 32) {
                cached_base = lp;
                cached_page = (lp + lane < n_pages) ? bt_row[lp + lane] : 0;
            }
            const int page = __shfl_sync(0xffffffffu, cached_page, lp - cached_base);
            if (lane == 0) {
                const int slot0 = page * P;
#pragma unroll
                for (int h = 0; h < kHalves; ++h) {
                    const int off = h * kBN * 128 + i * P * 128;
                    tma_load_3d(kdst + off, &tmap_k, h * 64, kvh, slot0, &bars[kBarKvFull + st],
                                policy);
                    tma_load_3d(vdst + off, &tmap_v, h * 64, kvh, slot0, &bars[kBarKvFull + st],
                                policy);
                }
            }
        }
        issued = b + 1;
    };
    if (warp == 0) {
        if (lane == 0) {
            for (int i = 0; i < kBarCount; ++i)
                mbar_init(&bars[i],
                          (i == kBarSFree || i == kBarPFull || i == kBarPFull + 1) ? 128u : 1u);
            fence_mbar_init();
            prefetch_tensormap(&tmap_q);
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
            // the tile's 128 / G tokens x G heads of this kv head, token-major
            mbar_arrive_expect_tx(&bars[kBarQFull], Geom::kQBytes);
#pragma unroll
            for (int h = 0; h < kHalves; ++h)
                tma_load_4d(sQ + h * kM * 128, &tmap_q, h * 64, 0, kvh, tok0 + row_begin / G,
                            &bars[kBarQFull]);
        }
        __syncwarp();
        policy = l2_policy_evict_last();   // the sibling row tile re-reads these pages
        for (int b = 0; b < min(kStages, n_blocks); ++b)
            produce_block(b);
    }
    if (warp == 1)
        tmem_alloc(tmem_slot, Geom::kTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_o = tmem;
    const uint32_t tmem_s = tmem + Geom::kColS;
    const uint32_t tmem_p = tmem + Geom::kColP;   // buffer j at tmem_p + 32 j
    bool ok = true;

    if (warp == 0) {
        // ------------------------------ TMA producer -------------------------------------
        for (int b = kStages; b < n_blocks; ++b) {
            const int st = b % kStages;
            const bool waited = mbar_wait(&bars[kBarKvEmpty + st], ((b / kStages) - 1) & 1);
            if (!__all_sync(0xffffffffu, waited)) {
                ok = false;
                break;
            }
            produce_block(b);
        }
        if (!ok && lane == 0) {
            atomicOr(&g_append_tc_errors, kErrAppendTcWait);
            for (int b = max(0, issued - kStages); b < issued; ++b)
                if (!mbar_wait(&bars[kBarKvFull + b % kStages], (b / kStages) & 1))
                    atomicOr(&g_append_tc_errors, kErrDrainWait);
            if (!mbar_wait(&bars[kBarQFull], 0))
                atomicOr(&g_append_tc_errors, kErrDrainWait);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ---------------------------------------
        constexpr uint32_t kIdescQK = umma_idesc_bf16(kM, kBN, 0);
        constexpr uint32_t kIdescPV = umma_idesc_bf16(kM, D, 1);
        const uint32_t q_addr = smem_addr(sQ);
        const uint32_t stage_addr = smem_addr(sStages);

        auto wait_all = [&](uint64_t *bar, uint32_t parity) {
            const bool w = mbar_wait(bar, parity);
            return __all_sync(0xffffffffu, w);
        };
        // Zero V rows n_valid .. kBN-1 of stage st (positions past the last visible one).
        auto zero_v_tail = [&](int st, int n_valid) {
            uint8_t *vt = sStages + st * Geom::kStageBytes + Geom::kTileBytes;
            const int rows_to_zero = kBN - n_valid;
            for (int idx = lane; idx < rows_to_zero * kHalves * 8; idx += 32) {
                const int chunk = idx & 7;
                const int rest = idx >> 3;
                const int h = rest % kHalves;
                const int r = n_valid + rest / kHalves;
                *reinterpret_cast<uint4 *>(vt + h * kBN * 128 + r * 128 + chunk * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
        };
        auto issue_qk = [&](int st) {
            tc_fence_after_sync();
            if (lane == 0) {
                const uint32_t k_addr = stage_addr + st * Geom::kStageBytes;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t da =
                        umma_desc_sw128(q_addr + (k >> 2) * kM * 128 + (k & 3) * 32, 16, 1024);
                    const uint64_t db =
                        umma_desc_sw128(k_addr + (k >> 2) * kBN * 128 + (k & 3) * 32, 16, 1024);
                    umma_bf16_ss(tmem_s, da, db, kIdescQK, k > 0 ? 1u : 0u);
                }
                umma_commit(&bars[kBarSFull]);
            }
            __syncwarp();
        };

        if (!wait_all(&bars[kBarQFull], 0))
            ok = false;
        // Event loop: issue whichever of QK_{next_qk} (needs its K/V stage and the softmax
        // warps to have read the previous S) and PV_{next_pv} (needs P) is ready first, so
        // the PV product of a block never waits for the next block's loads.
        int next_qk = 0, next_pv = 0;
        long long idle_since = clock64();
        while (ok && next_pv < n_blocks) {
            bool progressed = false;
            if (next_qk < n_blocks) {
                const int st = next_qk % kStages;
                bool ready = mbar_test(&bars[kBarKvFull + st], (next_qk / kStages) & 1) &&
                             (next_qk == 0 || mbar_test(&bars[kBarSFree], (next_qk - 1) & 1));
                ready = __shfl_sync(0xffffffffu, ready, 0);
                if (ready) {
                    const int n_valid = n_keys - next_qk * kBN;
                    if (n_valid < kBN)
                        zero_v_tail(st, n_valid);
                    issue_qk(st);
                    ++next_qk;
                    progressed = true;
                }
            }
            if (next_pv < next_qk) {
                bool ready = mbar_test(&bars[kBarPFull + (next_pv & 1)], (next_pv >> 1) & 1);
                ready = __shfl_sync(0xffffffffu, ready, 0);
                if (ready) {
                    const int st = next_pv % kStages;
                    tc_fence_after_sync();
                    if (lane == 0) {
                        const uint32_t v_addr =
                            stage_addr + st * Geom::kStageBytes + Geom::kTileBytes;
                        const uint32_t p_cols = tmem_p + (next_pv & 1) * 32;
#pragma unroll
                        for (int k = 0; k < kBN / 16; ++k) {
                            const uint64_t db =
                                umma_desc_sw128(v_addr + k * 16 * 128, kBN * 128, 1024);
                            umma_bf16_ts(tmem_o, p_cols + k * 8, db, kIdescPV,
                                         (next_pv > 0 || k > 0) ? 1u : 0u);
                        }
                        umma_commit(&bars[kBarPvDone + (next_pv & 1)]);
                        umma_commit(&bars[kBarKvEmpty + st]);
                    }
                    __syncwarp();
                    ++next_pv;
                    progressed = true;
                }
            }
            if (progressed) {
                idle_since = clock64();
            } else if (clock64() - idle_since > kWaitLimitCycles) {
                ok = false;
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        if (!ok && lane == 0)
            atomicOr(&g_append_tc_errors, kErrAppendTcWait);
        // Every MMA this thread issued must be complete before TMEM is released.
        if (lane == 0) {
            umma_commit(&bars[kBarDrain]);
            if (!mbar_wait(&bars[kBarDrain], 0))
                atomicOr(&g_append_tc_errors, kErrDrainWait);
        }
        __syncwarp();
    } else {
        // ------------------------------ softmax warps ------------------------------------
        const int quad = warp & 3;                  // TMEM lane quarter this warp may access
        const int row = quad * 32 + lane;           // row of the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const int gr = row_begin + row;
        const bool valid = gr < rows;
        const int ti = gr / G;
        const int lim = valid ? ctx - q_len + ti : -1;   // last visible position
        const float sl2 = a.scale_log2;
        float m_used = -INFINITY;
        float l_sum = 0.0f;

        for (int b = 0; b < n_blocks; ++b) {
            if (!__all_sync(0xffffffffu, mbar_wait(&bars[kBarSFull], b & 1))) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            float x[64];
            {
                float t0[32], t1[32];
                tmem_ld32(tmem_s + lane_off, t0);
                tmem_ld32(tmem_s + lane_off + 32, t1);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    x[c] = t0[c];
                    x[32 + c] = t1[c];
                }
            }
            tc_fence_before_sync();
            mbar_arrive(&bars[kBarSFree]);

            const int key0 = b * kBN;
            // causal limit (and positions past the loaded range) on the raw scores
            if (key0 + kBN - 1 > lim) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (key0 + c > lim)
                        x[c] = -INFINITY;
            }
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 64; ++c)
                mx = fmaxf(mx, x[c]);
            const float mb = mx * sl2;   // base-2 scaled row max of this block (scale > 0)
            // lazy rescale: move the reference max only when it grows by more than 2^8
            float alpha = 1.0f;
            bool moved = false;
            if (mb > m_used + kRescaleLog2) {
                alpha = (m_used == -INFINITY) ? 0.0f : fast_exp2(m_used - mb);
                m_used = mb;
                moved = true;
            }
            const float neg_mu = (m_used == -INFINITY) ? 0.0f : -m_used;
            uint32_t pk[32];
            float psum = 0.0f;
            if (__any_sync(0xffffffffu, valid)) {
                // p = 2^(s * scale * log2(e) - m); every fourth column on the FMA pipe
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float e0 = fast_exp2(fmaf(x[2 * c], sl2, neg_mu));
                    const float y1 = fmaf(x[2 * c + 1], sl2, neg_mu);
                    const float e1 = (c & 1) ? exp2_fma(y1) : fast_exp2(y1);
                    pk[c] = pack_bf16x2(e0, e1);
                    psum += bf16x2_sum(pk[c]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 32; ++c)   // a warp of padding rows: P = 0
                    pk[c] = 0u;
            }
            l_sum = l_sum * alpha + psum;

            // P buffer b & 1 was last read by PV(b - 2); O may be rescaled only once PV(b - 1)
            // is done.
            const int pb = b & 1;
            if (b >= 2 && !__all_sync(0xffffffffu, mbar_wait(&bars[kBarPvDone + pb],
                                                             ((b >> 1) - 1) & 1))) {
                ok = false;
                break;
            }
            if (b > 0 && __any_sync(0xffffffffu, moved)) {
                if (!__all_sync(0xffffffffu, mbar_wait(&bars[kBarPvDone + ((b - 1) & 1)],
                                                       ((b - 1) >> 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                {
                    const float f = moved ? alpha : 1.0f;
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        float o[32];
                        tmem_ld32(tmem_o + lane_off + c0, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            o[c] *= f;
                        tmem_st32(tmem_o + lane_off + c0, o);
                    }
                    tmem_wait_st();
                }
            }
            tc_fence_after_sync();
            // P row -> TMEM buffer pb: column j holds positions 2j, 2j + 1
            tmem_st32u(tmem_p + pb * 32 + lane_off, pk);
            tmem_wait_st();
            tc_fence_before_sync();
            mbar_arrive(&bars[kBarPFull + pb]);
        }

        // epilogue: O row / l -> global, once the last PV product is done
        if (ok && !__all_sync(0xffffffffu, mbar_wait(&bars[kBarPvDone + ((n_blocks - 1) & 1)],
                                                     ((n_blocks - 1) >> 1) & 1)))
            ok = false;
        tc_fence_after_sync();
        if (!ok)
            atomicOr(&g_append_tc_errors, kErrAppendTcWait);
        const float inv = (l_sum > 0.0f) ? 1.0f / l_sum : 0.0f;
        if (a.out_f32) {
            const int g = gr - ti * G;
            const size_t out_row =
                (static_cast<size_t>(tok0 + ti) * a.q_heads + static_cast<size_t>(kvh) * G + g) *
                D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                float o[32];
                tmem_ld32(tmem_o + lane_off + c0, o);
                tmem_wait_ld();
                if (valid && ok) {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(a.out) +
                                                             out_row + c0);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        dst[c] = make_float4(o[4 * c] * inv, o[4 * c + 1] * inv,
                                             o[4 * c + 2] * inv, o[4 * c + 3] * inv);
                }
            }
        } else {
            // Stage the bf16 tile in the query buffer (dead since the last QK product): row r
            // holds D * 2 bytes, 16-byte chunk c at (c & ~7) | ((c & 7) ^ (r & 7)), so eight
            // consecutive rows hit distinct banks.  Then store whole rows, coalesced.
            constexpr int kChunks = D / 8;
            uint8_t *stage_row = sQ + row * (D * 2);
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                float o[32];
                tmem_ld32(tmem_o + lane_off + c0, o);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int chunk = c0 / 8 + c;
                    const int phys = (chunk & ~7) | ((chunk & 7) ^ (row & 7));
                    *reinterpret_cast<uint4 *>(stage_row + phys * 16) =
                        make_uint4(pack_bf16x2(o[8 * c] * inv, o[8 * c + 1] * inv),
                                   pack_bf16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                   pack_bf16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                                   pack_bf16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
                }
            }
            named_barrier(1, 128);
            const int n_rows = min(kM, rows - row_begin);
            const int t = threadIdx.x - 64;   // 0 .. 127 over the softmax warps
            for (int idx = t; ok && idx < n_rows * kChunks; idx += 128) {
                const int r = idx / kChunks;
                const int chunk = idx - r * kChunks;
                const int phys = (chunk & ~7) | ((chunk & 7) ^ (r & 7));
                const int grr = row_begin + r;
                const int tok = grr / G;
                const size_t dst_row = (static_cast<size_t>(tok0 + tok) * a.q_heads +
                                        static_cast<size_t>(kvh) * G + (grr - tok * G)) * D;
                *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + dst_row +
                                           chunk * 8) =
                    *reinterpret_cast<const uint4 *>(sQ + r * (D * 2) + phys * 16);
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, Geom::kTmemCols);
    }
}

template <int D>
cudaError_t launch_t(const AppendLaunch &l, const CUtensorMap &tq, const CUtensorMap &tk,
                     const CUtensorMap &tv, cudaStream_t stream)
{
    Args a;
    a.out = l.out;
    a.out_f32 = l.out_f32;
    a.block_table = l.block_table;
    a.bt_stride = l.bt_stride;
    a.q_indptr = l.q_indptr;
    a.context_lens = l.context_lens;
    a.q_heads = l.q_heads;
    a.group = l.q_heads / l.kv_heads;
    a.page_size = l.page_size;
    a.scale_log2 = l.scale * kLog2e;
    const size_t smem = TcGeom<D>::kSmemBytes;
    auto kernel = paged_append_tc_kernel<D>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess)
        return err;
    const int tiles = (l.max_q_len * a.group + kM - 1) / kM;
    dim3 grid(tiles, l.kv_heads, l.num_seqs);
    kernel<<<grid, kThreads, smem, stream>>>(tq, tk, tv, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append_tc(const AppendLaunch &l, const CUtensorMap &tmap_q,
                             const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                             cudaStream_t stream)
{
    if (l.num_seqs == 0 || l.num_tokens == 0 || l.max_q_len == 0)
        return cudaSuccess;
    return l.head_dim == 128 ? launch_t<128>(l, tmap_q, tmap_k, tmap_v, stream)
                             : launch_t<64>(l, tmap_q, tmap_k, tmap_v, stream);
}

cudaError_t read_and_clear_append_tc_errors(uint32_t *flags)
{
    uint32_t zero = 0;
    cudaError_t err = cudaMemcpyFromSymbol(flags, g_append_tc_errors, sizeof(uint32_t));
    if (err != cudaSuccess)
        return err;
    return cudaMemcpyToSymbol(g_append_tc_errors, &zero, sizeof(uint32_t));
}

}  // namespace kvc
