// kvc_append_int8.cu -- causal chunked prefill over INT8 pages on the tcgen05 tensor cores.
//
// What it computes: kvc_append's attention (Quail "KV", "KV rewind"; TileInfer.jl "KV cache",
// "Prefix reuse in chat") over pages of int8 codes with one fp32 scale per (position, kv head)
// vector (TileInfer.jl "KV cache", "INT8 cache").  The cache is not dequantised: a key's scale
// multiplies its score and a value's scale its probability before the PV product; the codes
// themselves are the tensor-core operands.
//
// The tensor cores take 16-bit operands from shared memory, so codes pass through a
// conversion stage; both conversions are exact (|code| <= 128).  K codes become bf16, the
// bf16 query's type (a byte permute, two logic operations and one bf16x2 subtract per pair).
// V codes become fp16 (one xor, a byte permute and an fp16x2 subtract per pair) because the
// other operand of PV, P' = p * v_scale, is written as fp16: its 11-bit significand keeps the
// rounding of P' (and with it the error of a short context's output) four times below bf16's.
// fp16's range bounds P': p <= 2^4 (the running max lags the true one by at most 2^4) and a
// value scale above 4000 (|v| above 5.08e5) sets kErrScaleRange.
//
// Structure: kvc_append_tc.cu's (persistent, one CTA per SM; a work item is a pair of 128-row
// tiles of one (sequence, kv head); fixed-order MMA issue; P in TMEM over S's columns), head_dim
// 128, 14 warps:
//   warp 0      TMA: int8 code half-slots of 64 positions (one box per page) through a 7-deep
//               ring, in the order K(0), K(1), V(0), K(2), V(1), ..., and for each block the K
//               and V scale runs (one bulk copy each per page) into a 6-deep scale ring;
//   warp 1      TMEM and the MMA issue: S_t = Q_t K(b)^T (bf16) and O_t += P'_t V(b) (fp16);
//   warps 2, 3, 12, 13   converters 0-3: converter v turns rows 32 (v / 2) .. + 31 of code
//               half-slot v % 2 of each block into rows 64 (v % 2) + 32 (v / 2) .. of a 16-bit
//               operand slot (two K slots, one V slot, the MMA's 128-byte-swizzled
//               [half][128 positions][64 dims]); converter t < 2 also loads query tile t of
//               each item, and converter 0 readies each block's scales (K scales times
//               scale * log2(e), positions the item never sees set to 0);
//   warps 4-7   softmax of tile 0, warps 8-11 of tile 1: x = S * k_scale' with the causal
//               limit, lazy running max, p = 2^(x - m), P' = p * v_scale as fp16 pairs into TMEM.
// The single V slot is released as soon as the last tile's PV product of a block is done; the
// next V is converted while the softmax works on the S of the block after.  The softmax
// denominator sums p (before the value scale).  A position the item never sees may hold any
// codes and a NaN scale: its scales are replaced by 0 before the softmax reads them, its scores
// are masked, and its operand rows are finite codes or never read.
#include <math.h>

#include "kvc_append_items.cuh"
#include "kvc_device.cuh"
#include "kvc_launch.h"

namespace kvc {

namespace {

__device__ uint32_t g_append_int8_errors;

using append::Item;
using append::kBN;
using append::kM;
using append::seq_of;
using append::Walker;

constexpr int kThreads = 14 * 32;
constexpr int kConverters = 4;
constexpr int kCodeSlots = 7;              // 64-position code half-slots
constexpr int kScaleSlots = 6;             // blocks of K and V scales
constexpr int kHalfRows = kBN / 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 4.0f;
constexpr float kMaxValueScale = 4000.0f;   // 2^4 * 4000 < 65504, fp16's largest value

constexpr int kScaleBytes = 2 * kBN * 4;          // K scales, then V scales, of one block
constexpr uint32_t kTmemCols = 512;

// Shared memory for head_dim D (64 or 128): query tiles, operand slots, code slots, scales.
template <int D>
struct A8Geom {
    static constexpr int kHalves = D / 64;                 // 64-dim halves of a 16-bit row
    static constexpr int kQBytes = kHalves * kM * 128;     // one bf16 query tile
    static constexpr int kOpBytes = kHalves * kBN * 128;   // K or V of 128 positions, 16-bit
    static constexpr int kCodeBytes = kHalfRows * D;       // codes of 64 positions
    static constexpr int kOffOp = 2 * kQBytes;             // operand slots: K0, K1, V
    static constexpr int kOffCode = kOffOp + 3 * kOpBytes;
    static constexpr int kOffScale = kOffCode + kCodeSlots * kCodeBytes;
    static constexpr int kOffBar = kOffScale + kScaleSlots * kScaleBytes;
    static constexpr uint32_t kColS = D;   // TMEM per tile w at 256 w: O [0, D), S [D, D + 128)
};

enum BarIndex : int {
    kBarCodeFull = 0,
    kBarCodeEmpty = kBarCodeFull + kCodeSlots,     // the two converters of a half-slot
    kBarKFull = kBarCodeEmpty + kCodeSlots,        // [2], every converter
    kBarKEmpty = kBarKFull + 2,                    // [2], MMA commit
    kBarVFull = kBarKEmpty + 2,                    // every converter
    kBarVEmpty = kBarVFull + 1,                    // MMA commit
    kBarScaleFull = kBarVEmpty + 1,
    kBarScaleReady = kBarScaleFull + kScaleSlots,  // converter warp 2
    kBarScaleEmpty = kBarScaleReady + kScaleSlots, // one arrival per softmax warp (8)
    kBarQFull = kBarScaleEmpty + kScaleSlots,      // [tile]
    kBarQEmpty = kBarQFull + 2,                    // [tile], MMA commit after its last S product
    kBarSFull = kBarQEmpty + 2,                    // [tile]
    kBarPFull = kBarSFull + 2,                     // [tile], 128 arrivals
    kBarPvDone = kBarPFull + 2,                    // [tile]
    kBarDrain = kBarPvDone + 2,
    kBarCount
};
template <int D>
constexpr size_t a8_smem_bytes()
{
    return A8Geom<D>::kOffBar + kBarCount * 8 + 16;
}
static_assert(a8_smem_bytes<128>() <= 232448 && a8_smem_bytes<64>() <= 232448, "shared memory");

struct Args {
    void *out;
    int out_f32;
    const float *k_scales, *v_scales;
    const int32_t *block_table;
    int bt_stride;
    const int32_t *q_indptr;
    const int32_t *context_lens;
    int kv_heads, q_heads, group, page_size, pairs_per_seq, num_items;
    float scale_log2;
    uint32_t *err;   // the caller's device error word, or null (this file's own word)
    int hnd;         // HND codes: page boxes addressed by (offset, page * kv_heads + kv head)
};

// Fill order of an item's K / V blocks: j = 0 .. 2 nb - 1 is K(0), K(1), V(0), K(2), V(1), ...,
// V(nb - 1), so V(b) lands next to K(b + 1), about when PV(b) needs it.
__device__ __forceinline__ void block_of_fill(int j, int nb, bool &is_k, int &b)
{
    is_k = j == 0 || (j < 2 * nb - 1 && (j & 1));
    b = is_k ? (j + 1) / 2 : (j == 2 * nb - 1 ? nb - 1 : j / 2 - 1);
}

// Rows 0 .. rows - 1 (a multiple of 16, at most 64) of a 128-byte-swizzled slot of int8 codes
// [rows][128 dims] -> the same rows of a 16-bit operand slot [2 dim halves][128 rows][64 dims]
// (dst points at the first row of half 0; halves are kBN * 128 bytes apart).  K codes become
// bf16, V codes fp16.  One warp; lane (r0, c) = (lane / 8, lane % 8) converts dims
// 16 c .. 16 c + 15 of rows 4 k + r0; a row's swizzle phase (row mod 8) is r0 for even k and
// r0 + 4 for odd k, so each lane's offsets are two constants.
template <int D>
__device__ __forceinline__ void convert_rows(const uint8_t *src, uint8_t *dst, int rows,
                                             bool to_bf16, int lane);

template <>
__device__ __forceinline__ void convert_rows<128>(const uint8_t *src, uint8_t *dst, int rows,
                                                  bool to_bf16, int lane)
{
    const int r0 = lane >> 3;
    const int c = lane & 7;
    const int q0 = 2 * (c & 3);
    int src_off[2], dst_off0[2], dst_off1[2];
#pragma unroll
    for (int odd = 0; odd < 2; ++odd) {
        const int sw = r0 + 4 * odd;
        src_off[odd] = r0 * 128 + ((c ^ sw) << 4);
        dst_off0[odd] = (c >> 2) * kBN * 128 + r0 * 128 + ((q0 ^ sw) << 4);
        dst_off1[odd] = (c >> 2) * kBN * 128 + r0 * 128 + (((q0 + 1) ^ sw) << 4);
    }
    // steps of 16 rows: the four loads of a step are issued before its stores
#pragma unroll 1
    for (int s4 = 0; s4 < rows; s4 += 16) {
        const uint8_t *sp = src + s4 * 128;
        uint8_t *dp = dst + s4 * 128;
        uint4 cw[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            cw[k] = *reinterpret_cast<const uint4 *>(sp + 4 * k * 128 + src_off[k & 1]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t f[8];
            if (to_bf16) {
                codes_word_bf16x2(cw[k].x, f[0], f[1]);
                codes_word_bf16x2(cw[k].y, f[2], f[3]);
                codes_word_bf16x2(cw[k].z, f[4], f[5]);
                codes_word_bf16x2(cw[k].w, f[6], f[7]);
            } else {
                codes_word_f16x2(cw[k].x, f[0], f[1]);
                codes_word_f16x2(cw[k].y, f[2], f[3]);
                codes_word_f16x2(cw[k].z, f[4], f[5]);
                codes_word_f16x2(cw[k].w, f[6], f[7]);
            }
            *reinterpret_cast<uint4 *>(dp + 4 * k * 128 + dst_off0[k & 1]) =
                make_uint4(f[0], f[1], f[2], f[3]);
            *reinterpret_cast<uint4 *>(dp + 4 * k * 128 + dst_off1[k & 1]) =
                make_uint4(f[4], f[5], f[6], f[7]);
        }
    }
}

// The same for head_dim 64: code rows of 64 bytes under the 64-byte swizzle (16-byte chunk c
// of row r at c ^ ((r / 2) % 4)) -> rows of a one-half operand slot [128 rows][64 dims].  Lane
// (r0, c) = (lane / 4, lane % 4) converts dims 16 c .. 16 c + 15 of rows 8 k + r0 (output
// chunks 2 c and 2 c + 1 of the row, 128-byte swizzle); both loads of a step issue before the
// stores.
template <>
__device__ __forceinline__ void convert_rows<64>(const uint8_t *src, uint8_t *dst, int rows,
                                                 bool to_bf16, int lane)
{
    const int r0 = lane >> 2;
    const int c = lane & 3;
#pragma unroll 1
    for (int s4 = 0; s4 < rows; s4 += 16) {
        uint4 cw[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int row = s4 + 8 * k + r0;
            cw[k] = *reinterpret_cast<const uint4 *>(src + row * 64 +
                                                     ((c ^ ((row >> 1) & 3)) << 4));
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int row = s4 + 8 * k + r0;
            uint32_t f[8];
            if (to_bf16) {
                codes_word_bf16x2(cw[k].x, f[0], f[1]);
                codes_word_bf16x2(cw[k].y, f[2], f[3]);
                codes_word_bf16x2(cw[k].z, f[4], f[5]);
                codes_word_bf16x2(cw[k].w, f[6], f[7]);
            } else {
                codes_word_f16x2(cw[k].x, f[0], f[1]);
                codes_word_f16x2(cw[k].y, f[2], f[3]);
                codes_word_f16x2(cw[k].z, f[4], f[5]);
                codes_word_f16x2(cw[k].w, f[6], f[7]);
            }
            uint8_t *out = dst + row * 128;
            const int sw = row & 7;
            *reinterpret_cast<uint4 *>(out + (((2 * c) ^ sw) << 4)) =
                make_uint4(f[0], f[1], f[2], f[3]);
            *reinterpret_cast<uint4 *>(out + (((2 * c + 1) ^ sw) << 4)) =
                make_uint4(f[4], f[5], f[6], f[7]);
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    paged_append_int8_kernel(const __grid_constant__ CUtensorMap tmap_q,
                             const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v, const Args a)
{
    pdl_wait();
    pdl_trigger();
    using Geom = A8Geom<D>;
    constexpr int kHalves = Geom::kHalves, kQBytes = Geom::kQBytes, kOpBytes = Geom::kOpBytes;
    constexpr int kCodeBytes = Geom::kCodeBytes, kOffOp = Geom::kOffOp;
    constexpr int kOffCode = Geom::kOffCode, kOffScale = Geom::kOffScale;
    constexpr int kOffBar = Geom::kOffBar;
    constexpr uint32_t kColS = Geom::kColS;
    extern __shared__ __align__(1024) uint8_t smem[];
    if ((smem_addr(smem) & 1023u) != 0) {
        if (threadIdx.x == 0)
            atomicOr(a.err ? a.err : &g_append_int8_errors, kErrSmemAlign);
        return;
    }
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kBarCount);
    auto q_tile = [&](int tile) { return smem + tile * kQBytes; };
    // operand slot of K number nk (two slots, alternating); V has one slot
    auto k_op = [&](int nk) { return smem + kOffOp + (nk & 1) * kOpBytes; };
    uint8_t *v_op = smem + kOffOp + 2 * kOpBytes;
    auto code_slot = [&](int m) { return smem + kOffCode + (m % kCodeSlots) * kCodeBytes; };
    auto scale_slot = [&](int sb) {
        return reinterpret_cast<float *>(smem + kOffScale + (sb % kScaleSlots) * kScaleBytes);
    };
    uint32_t *err = a.err ? a.err : &g_append_int8_errors;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.group;
    const int P = a.page_size;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kBarCount; ++i) {
            uint32_t count = 1;
            if (i == kBarKFull || i == kBarKFull + 1 || i == kBarVFull)
                count = kConverters;
            else if (i >= kBarCodeEmpty && i < kBarCodeEmpty + kCodeSlots)
                count = 2;
            else if (i >= kBarScaleEmpty && i < kBarScaleEmpty + kScaleSlots)
                count = 8;
            else if (i == kBarPFull || i == kBarPFull + 1)
                count = 128;
            mbar_init(&bars[i], count);
        }
        fence_mbar_init();
    }
    if (warp == 1)
        tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        // ------------------------------ codes and scales ----------------------------------
        if (lane == 0) {
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
        }
        const uint64_t policy = l2_policy_evict_first();
        const int pages_per_half = kHalfRows / P;
        Walker w;
        w.start(a, err);
        int m = 0;    // code half-slots filled so far (two per K / V block)
        int sb = 0;   // scale blocks filled so far
        while (ok && !w.done) {
            const Item &x = w.x;
            const int32_t *bt_row = a.block_table + static_cast<size_t>(x.s) * a.bt_stride;
            const int n_pages = (x.n_keys + P - 1) / P;
            int cached_base = -64;
            int cached_page = 0;
            const int nb = x.n_blocks;
            for (int j = 0; j < 2 * nb && ok; ++j) {
                bool is_k;
                int b;
                block_of_fill(j, nb, is_k, b);
                const int key0 = b * kBN;
                const int np = (min(kBN, x.n_keys - key0) + P - 1) / P;
                const int lp0 = key0 / P;   // first page of the block
                if (lp0 < cached_base || lp0 + np > cached_base + 32) {
                    cached_base = lp0;
                    cached_page = (lp0 + lane < n_pages) ? bt_row[lp0 + lane] : 0;
                }
                for (int h = 0; h < 2; ++h) {
                    const int cs = m % kCodeSlots;
                    if (m >= kCodeSlots &&
                        !__all_sync(0xffffffffu, mbar_wait(&bars[kBarCodeEmpty + cs],
                                                           ((m / kCodeSlots) - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    const bool scales = is_k && h == 0;
                    const int ss = sb % kScaleSlots;
                    if (scales && sb >= kScaleSlots &&
                        !__all_sync(0xffffffffu, mbar_wait(&bars[kBarScaleEmpty + ss],
                                                           ((sb / kScaleSlots) - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    // pages h * pages_per_half .. of the block that exist (none: the half-slot
                    // completes on the arrival alone)
                    const int np_h = min(max(np - h * pages_per_half, 0), pages_per_half);
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&bars[kBarCodeFull + cs],
                                              static_cast<uint32_t>(np_h * P * D));
                        if (scales)
                            mbar_arrive_expect_tx(&bars[kBarScaleFull + ss],
                                                  static_cast<uint32_t>(np * P * 4 * 2));
                    }
                    __syncwarp();
                    // lanes 0 .. np_h - 1: code boxes of the half's pages; with the scales,
                    // lane 8 + 2 i + op: page i's K (op 0) or V (op 1) scale run
                    const int i = lane < 8 ? h * pages_per_half + lane : (lane - 8) >> 1;
                    const int page =
                        __shfl_sync(0xffffffffu, cached_page, (lp0 - cached_base + i) & 31);
                    if (lane < np_h) {
                        tma_load_3d(code_slot(m) + lane * P * D, is_k ? &tmap_k : &tmap_v, 0,
                                    a.hnd ? 0 : x.kvh, a.hnd ? page * a.kv_heads + x.kvh : page * P,
                                    &bars[kBarCodeFull + cs], policy);
                    } else if (scales && lane >= 8 && i < np) {
                        const int op = (lane - 8) & 1;
                        const float *src = (op == 0 ? a.k_scales : a.v_scales) +
                                           (static_cast<size_t>(page) * a.kv_heads + x.kvh) * P;
                        bulk_load(reinterpret_cast<uint8_t *>(scale_slot(sb)) + op * kBN * 4 +
                                      i * P * 4,
                                  src, static_cast<uint32_t>(P * 4), &bars[kBarScaleFull + ss]);
                    }
                    ++m;
                    if (scales)
                        ++sb;
                }
            }
            if (!ok)
                break;
            w.next(a, err);
        }
        if (!ok && lane == 0) {
            atomicOr(err, kErrAppendTcWait);
            // let every copy in flight land before the CTA can exit
            for (int k = max(0, m - kCodeSlots); k < m; ++k)
                if (!mbar_wait(&bars[kBarCodeFull + k % kCodeSlots], (k / kCodeSlots) & 1))
                    atomicOr(err, kErrDrainWait);
            for (int k = max(0, sb - kScaleSlots); k < sb; ++k)
                if (!mbar_wait(&bars[kBarScaleFull + k % kScaleSlots], (k / kScaleSlots) & 1))
                    atomicOr(err, kErrDrainWait);
        }
    } else if (warp == 2 || warp == 3 || warp >= 12) {
        // ------------------------------ converters and query loads -----------------------
        const int cv = warp < 12 ? warp - 2 : warp - 10;   // converter 0 .. 3
        const int h = cv & 1;      // code half-slot / operand rows 64 h ..; query tile h
        const int sub = cv >> 1;   // rows 32 sub .. 32 sub + 31 of the half
        if (lane == 0)
            prefetch_tensormap(&tmap_q);
        Walker w;
        w.start(a, err);
        int n = 0, nk = 0, nv = 0, sb = 0;
        int qi = 0;   // items whose query tile h was requested
        while (ok && !w.done) {
            const Item &x = w.x;
            const int nb = x.n_blocks;
            if (sub == 0 && (h == 0 || x.has_b)) {
                // query tile h of this item, once its last S product of the previous item is done
                if (qi > 0 && !__all_sync(0xffffffffu,
                                          mbar_wait(&bars[kBarQEmpty + h], (qi - 1) & 1))) {
                    ok = false;
                    break;
                }
                if (lane == 0)
                    mbar_arrive_expect_tx(&bars[kBarQFull + h], static_cast<uint32_t>(kQBytes));
                __syncwarp();
                if (lane < kHalves)
                    tma_load_4d(q_tile(h) + lane * kM * 128, &tmap_q, lane * 64, 0, x.kvh,
                                x.tok0 + (x.row_begin + h * kM) / G, &bars[kBarQFull + h]);
                ++qi;
            }
            const int last_cols = ((x.n_keys - (nb - 1) * kBN) + 15) & ~15;
            for (int j = 0; j < 2 * nb; ++j, ++n) {
                bool is_k;
                int b;
                block_of_fill(j, nb, is_k, b);
                const int m = 2 * n + h;
                uint64_t *full_bar;
                uint8_t *dst;
                bool waited;
                if (is_k) {
                    waited = nk < 2 || __all_sync(0xffffffffu,
                                                  mbar_wait(&bars[kBarKEmpty + (nk & 1)],
                                                            ((nk >> 1) - 1) & 1));
                    full_bar = &bars[kBarKFull + (nk & 1)];
                    dst = k_op(nk);
                    ++nk;
                } else {
                    waited = nv < 1 || __all_sync(0xffffffffu,
                                                  mbar_wait(&bars[kBarVEmpty], (nv - 1) & 1));
                    full_bar = &bars[kBarVFull];
                    dst = v_op;
                    ++nv;
                }
                if (!waited || !__all_sync(0xffffffffu,
                                           mbar_wait(&bars[kBarCodeFull + m % kCodeSlots],
                                                     (m / kCodeSlots) & 1))) {
                    ok = false;
                    break;
                }
                if (is_k && cv == 0) {
                    // scales of block b: K scales times scale * log2(e); 0 past the item's keys
                    const int ss = sb % kScaleSlots;
                    if (!__all_sync(0xffffffffu, mbar_wait(&bars[kBarScaleFull + ss],
                                                           (sb / kScaleSlots) & 1))) {
                        ok = false;
                        break;
                    }
                    float *sc = scale_slot(sb);
                    const int n_in = x.n_keys - b * kBN;
                    bool range_ok = true;
#pragma unroll
                    for (int e = 0; e < 2 * kBN / 32; ++e) {
                        const int idx = lane + 32 * e;
                        const bool live = (idx & (kBN - 1)) < n_in;
                        const float v = live ? sc[idx] : 0.0f;
                        if (idx >= kBN && !(v <= kMaxValueScale))
                            range_ok = false;
                        sc[idx] = idx < kBN ? v * a.scale_log2 : v;
                    }
                    if (!range_ok)
                        atomicOr(err, kErrScaleRange);
                    fence_proxy_async_smem();   // the next bulk copy into this slot
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&bars[kBarScaleReady + ss]);
                    ++sb;
                }
                // rows of this half that the products read (the last block: up to a multiple
                // of 16 past its last position; the codes there are loaded and finite)
                const int cols = (b + 1 == nb) ? last_cols : kBN;
                const int r_lo = h * kHalfRows + sub * (kHalfRows / 2);
                const int rows = min(max(cols - r_lo, 0), kHalfRows / 2);
                convert_rows<D>(code_slot(m) + sub * (kHalfRows / 2) * D, dst + r_lo * 128,
                                rows, is_k, lane);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(full_bar);
                    mbar_arrive(&bars[kBarCodeEmpty + m % kCodeSlots]);
                }
            }
            if (!ok)
                break;
            w.next(a, err);
        }
        if (!ok && lane == 0) {
            atomicOr(err, kErrAppendTcWait);
            if (sub == 0 && qi > 0 && !mbar_wait(&bars[kBarQFull + h], (qi - 1) & 1))
                atomicOr(err, kErrDrainWait);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issue ----------------------------------------
        constexpr uint32_t kIdescPV = umma_idesc_f16(kM, D, 1);
        auto issue_qk = [&](int t, uint32_t k_addr, int n_cols) {
            const uint32_t idesc = umma_idesc_bf16(kM, n_cols, 0);
            const uint32_t q_addr = smem_addr(q_tile(t));
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint64_t da =
                    umma_desc_sw128(q_addr + (k >> 2) * kM * 128 + (k & 3) * 32, 16, 1024);
                const uint64_t db =
                    umma_desc_sw128(k_addr + (k >> 2) * kBN * 128 + (k & 3) * 32, 16, 1024);
                umma_bf16_ss(tmem + t * 256 + kColS, da, db, idesc, k > 0 ? 1u : 0u);
            }
        };
        auto issue_pv = [&](int t, uint32_t v_addr, int k_steps, bool first) {
            for (int k = 0; k < k_steps; ++k) {
                const uint64_t db = umma_desc_sw128(v_addr + k * 16 * 128, kBN * 128, 1024);
                umma_bf16_ts(tmem + t * 256, tmem + t * 256 + kColS + k * 8, db, kIdescPV,
                             (!first || k > 0) ? 1u : 0u);
            }
        };
        auto wait_k = [&](int nk) {
            return __all_sync(0xffffffffu,
                              mbar_wait(&bars[kBarKFull + (nk & 1)], (nk >> 1) & 1));
        };
        const uint32_t v_addr = smem_addr(v_op);
        Walker w;
        w.start(a, err);
        int nk = 0, nv = 0;
        int qi[2] = {0, 0};
        int tb[2] = {0, 0};
        while (ok && !w.done) {
            const Item &x = w.x;
            const int nt = x.has_b ? 2 : 1;
            const int nb = x.n_blocks;
            const int last_cols = ((x.n_keys - (nb - 1) * kBN) + 15) & ~15;
            if (!wait_k(nk)) {
                ok = false;
                break;
            }
            for (int t = 0; t < nt && ok; ++t) {
                if (!__all_sync(0xffffffffu, mbar_wait(&bars[kBarQFull + t], qi[t] & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                if (lane == 0) {
                    issue_qk(t, smem_addr(k_op(nk)), nb == 1 ? last_cols : kBN);
                    umma_commit(&bars[kBarSFull + t]);
                    if (nb == 1)
                        umma_commit(&bars[kBarQEmpty + t]);
                }
                __syncwarp();
            }
            if (!ok)
                break;
            if (lane == 0)
                umma_commit(&bars[kBarKEmpty + (nk & 1)]);
            __syncwarp();
            ++nk;
            for (int b = 0; b < nb && ok; ++b) {
                const bool last = b + 1 == nb;
                if (!__all_sync(0xffffffffu, mbar_wait(&bars[kBarVFull], nv & 1))) {
                    ok = false;
                    break;
                }
                for (int t = 0; t < nt; ++t) {
                    if (!__all_sync(0xffffffffu, mbar_wait(&bars[kBarPFull + t], tb[t] & 1))) {
                        ok = false;
                        break;
                    }
                    ++tb[t];
                    tc_fence_after_sync();
                    if (lane == 0) {
                        issue_pv(t, v_addr, last ? last_cols / 16 : kBN / 16, b == 0);
                        if (t + 1 == nt)
                            umma_commit(&bars[kBarVEmpty]);   // V(b) read by every tile
                        if (last)
                            umma_commit(&bars[kBarPvDone + t]);
                    }
                    __syncwarp();
                    if (last)
                        continue;
                    // K(b + 1) is waited for only once PV(b) of tile 0 is on its way
                    if (t == 0 && !wait_k(nk)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    if (lane == 0) {
                        issue_qk(t, smem_addr(k_op(nk)), b + 2 == nb ? last_cols : kBN);
                        umma_commit(&bars[kBarSFull + t]);
                        if (b + 2 == nb)
                            umma_commit(&bars[kBarQEmpty + t]);
                    }
                    __syncwarp();
                }
                if (!ok)
                    break;
                ++nv;
                if (!last) {
                    if (lane == 0)
                        umma_commit(&bars[kBarKEmpty + (nk & 1)]);
                    __syncwarp();
                    ++nk;
                }
            }
            if (!ok)
                break;
            for (int t = 0; t < nt; ++t)
                ++qi[t];
            w.next(a, err);
        }
        if (!ok && lane == 0)
            atomicOr(err, kErrAppendTcWait);
        // Every MMA this thread issued must be complete before TMEM is released.
        if (lane == 0) {
            umma_commit(&bars[kBarDrain]);
            if (!mbar_wait(&bars[kBarDrain], 0))
                atomicOr(err, kErrDrainWait);
        }
        __syncwarp();
    } else {
        // ------------------------------ softmax + epilogue -------------------------------
        const int t = (warp - 4) >> 2;               // tile
        const int quad = warp & 3;                   // TMEM lanes 32 quad ..
        const int row = quad * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tmem_o = tmem + t * 256 + lane_off;
        const uint32_t tmem_s = tmem + t * 256 + kColS + lane_off;
        Walker w;
        w.start(a, err);
        int tb = 0;   // blocks of this tile
        int ti = 0;   // items of this tile
        int sb = 0;   // scale blocks of every item (both tile groups release each one)
        auto release_scales = [&](int s) {
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars[kBarScaleEmpty + s % kScaleSlots]);
        };
        for (; ok && !w.done; w.next(a, err)) {
            const Item &x = w.x;
            if (t == 1 && !x.has_b) {
                for (int b = 0; b < x.n_blocks; ++b, ++sb) {
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(&bars[kBarScaleReady + sb % kScaleSlots],
                                              (sb / kScaleSlots) & 1))) {
                        ok = false;
                        break;
                    }
                    release_scales(sb);
                }
                continue;
            }
            const int gr = x.row_begin + t * kM + row;
            const bool valid = gr < x.rows;
            const int tok = gr / G;
            const int lim = valid ? x.ctx - x.q_len + tok : -1;   // last visible position
            const bool warp_valid = __any_sync(0xffffffffu, valid);
            float m_used = -INFINITY;
            float l_sum = 0.0f;
            for (int b = 0; b < x.n_blocks; ++b, ++tb, ++sb) {
                if (!__all_sync(0xffffffffu, mbar_wait(&bars[kBarSFull + t], tb & 1)) ||
                    !__all_sync(0xffffffffu,
                                mbar_wait(&bars[kBarScaleReady + sb % kScaleSlots],
                                          (sb / kScaleSlots) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const float4 *ks4 = reinterpret_cast<const float4 *>(scale_slot(sb));
                const float4 *vs4 = ks4 + kBN / 4;
                const int n_vis = min(max(lim - b * kBN + 1, 0), kBN);
                float alpha = 1.0f;
                bool moved = false;
                if (warp_valid) {
                    // pass 1: x = S * k_scale * scale * log2(e), -inf where masked, back to
                    // TMEM; the row max.  Two 64-column halves (fewer live registers); paired
                    // multiplies by the key scales; masking only where a row of the warp sees
                    // fewer than 128 positions of this block.
                    auto scale_quad = [&](float *x4, const float4 k4) {
                        f2_unpack(f2_mul(f2_pack(x4[0], x4[1]), f2_pack(k4.x, k4.y)), x4[0],
                                  x4[1]);
                        f2_unpack(f2_mul(f2_pack(x4[2], x4[3]), f2_pack(k4.z, k4.w)), x4[2],
                                  x4[3]);
                    };
                    const bool full = __all_sync(0xffffffffu, n_vis == kBN);
                    float mx = -INFINITY;
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        float xs[2][32];
                        tmem_ld32(tmem_s + 64 * hh, xs[0]);
                        tmem_ld32(tmem_s + 64 * hh + 32, xs[1]);
                        tmem_wait_ld();
                        if (full) {
#pragma unroll
                            for (int c = 0; c < 2; ++c) {
#pragma unroll
                                for (int j4 = 0; j4 < 8; ++j4) {
                                    float *x4 = &xs[c][4 * j4];
                                    scale_quad(x4, ks4[16 * hh + 8 * c + j4]);
                                    mx = fmax3(mx, x4[0], x4[1]);
                                    mx = fmax3(mx, x4[2], x4[3]);
                                }
                            }
                        } else {
#pragma unroll
                            for (int c = 0; c < 2; ++c) {
#pragma unroll
                                for (int j4 = 0; j4 < 8; ++j4) {
                                    float *x4 = &xs[c][4 * j4];
                                    scale_quad(x4, ks4[16 * hh + 8 * c + j4]);
#pragma unroll
                                    for (int e = 0; e < 4; ++e)
                                        if (64 * hh + 32 * c + 4 * j4 + e >= n_vis)
                                            x4[e] = -INFINITY;
                                    mx = fmax3(mx, x4[0], x4[1]);
                                    mx = fmax3(mx, x4[2], x4[3]);
                                }
                            }
                        }
                        tmem_st32(tmem_s + 64 * hh, xs[0]);
                        tmem_st32(tmem_s + 64 * hh + 32, xs[1]);
                    }
                    tmem_wait_st();
                    if (mx > m_used + kRescaleLog2) {
                        alpha = (m_used == -INFINITY) ? 0.0f : fast_exp2(m_used - mx);
                        m_used = mx;
                        moved = true;
                    }
                }
                // O holds every earlier PV product: rescale it in place when the max moved
                if (b > 0 && __any_sync(0xffffffffu, moved)) {
                    const float f = moved ? alpha : 1.0f;
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        float o[32];
                        tmem_ld32(tmem_o + c0, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            o[j] *= f;
                        tmem_st32(tmem_o + c0, o);
                    }
                }
                // pass 2: p = 2^(x - m) on MUFU, the rest in paired arithmetic; P' = p * v_scale
                // as fp16 pairs over S columns [16 c, 16 c + 16), which hold only chunks already
                // read.  A masked x is -inf: its p is 0.
                const float neg_mu = (m_used == -INFINITY) ? 0.0f : -m_used;
                const uint64_t nm2 = f2_pack(neg_mu, neg_mu);
                uint64_t psum2 = f2_pack(0.0f, 0.0f);
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[16];
                    if (warp_valid) {
                        float v[32];
                        tmem_ld32(tmem_s + 32 * c, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int j8 = 0; j8 < 4; ++j8) {
                            const float *v8 = &v[8 * j8];
                            float e[8];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                f2_unpack(f2_add(f2_pack(v8[2 * q], v8[2 * q + 1]), nm2),
                                          e[2 * q], e[2 * q + 1]);
                                e[2 * q] = fast_exp2(e[2 * q]);
                                e[2 * q + 1] = fast_exp2(e[2 * q + 1]);
                            }
                            const float4 sa = vs4[8 * c + 2 * j8];
                            const float4 sb = vs4[8 * c + 2 * j8 + 1];
                            const float sv[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const uint64_t e2 = f2_pack(e[2 * q], e[2 * q + 1]);
                                psum2 = f2_add(psum2, e2);
                                float p0, p1;
                                f2_unpack(f2_mul(e2, f2_pack(sv[2 * q], sv[2 * q + 1])), p0, p1);
                                pk[4 * j8 + q] = pack_f16x2(p0, p1);
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j)   // a warp of padding rows: P' = 0
                            pk[j] = 0u;
                    }
                    tmem_st16u(tmem_s + 16 * c, pk);
                }
                float ps0, ps1;
                f2_unpack(psum2, ps0, ps1);
                const float psum = ps0 + ps1;
                l_sum = l_sum * alpha + psum;
                tmem_wait_st();
                tc_fence_before_sync();
                mbar_arrive(&bars[kBarPFull + t]);
                release_scales(sb);
            }
            if (!ok)
                break;
            // epilogue: once this tile's last PV is done, O / l -> global
            if (!__all_sync(0xffffffffu, mbar_wait(&bars[kBarPvDone + t], ti & 1))) {
                ok = false;
                break;
            }
            ++ti;
            tc_fence_after_sync();
            const float inv = (l_sum > 0.0f) ? 1.0f / l_sum : 0.0f;
            const int g = gr - tok * G;
            const size_t out_row =
                (static_cast<size_t>(x.tok0 + tok) * a.q_heads + static_cast<size_t>(x.kvh) * G +
                 g) * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                float o[32];
                tmem_ld32(tmem_o + c0, o);
                tmem_wait_ld();
                if (valid) {
                    if (a.out_f32) {
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(a.out) +
                                                                 out_row + c0);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[j] = make_float4(o[4 * j] * inv, o[4 * j + 1] * inv,
                                                 o[4 * j + 2] * inv, o[4 * j + 3] * inv);
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>(
                            static_cast<__nv_bfloat16 *>(a.out) + out_row + c0);
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            dst[c] = make_uint4(pack_bf16x2(o[8 * c] * inv, o[8 * c + 1] * inv),
                                                pack_bf16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                                pack_bf16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                                                pack_bf16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
                    }
                }
                __syncwarp();
            }
            tc_fence_before_sync();
        }
        if (!ok)
            atomicOr(err, kErrAppendTcWait);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

int sm_count()
{
    static int count = 0;
    if (count == 0) {
        int dev = 0, n = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
            count = n;
        else
            count = 152;
    }
    return count;
}

}  // namespace

cudaError_t launch_append_int8(const AppendInt8Launch &l, const CUtensorMap &tmap_q,
                               const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                               cudaStream_t stream)
{
    if (l.num_seqs == 0 || l.num_tokens == 0 || l.max_q_len == 0)
        return cudaSuccess;
    Args a;
    a.out = l.out;
    a.out_f32 = l.out_f32;
    a.k_scales = l.k_scales;
    a.v_scales = l.v_scales;
    a.block_table = l.block_table;
    a.bt_stride = l.bt_stride;
    a.q_indptr = l.q_indptr;
    a.context_lens = l.context_lens;
    a.kv_heads = l.kv_heads;
    a.q_heads = l.q_heads;
    a.group = l.q_heads / l.kv_heads;
    a.page_size = l.page_size;
    const int tiles = (l.max_q_len * a.group + kM - 1) / kM;
    a.pairs_per_seq = (tiles + 1) / 2;
    const long long items = static_cast<long long>(a.pairs_per_seq) * l.kv_heads * l.num_seqs;
    if (items > 0x7FFFFFFFLL)
        return cudaErrorInvalidValue;
    a.num_items = static_cast<int>(items);
    a.scale_log2 = l.scale * kLog2e;
    a.err = current_error_word();
    a.hnd = l.hnd ? 1 : 0;
    const bool d64 = l.head_dim == 64;
    auto kernel = d64 ? paged_append_int8_kernel<64> : paged_append_int8_kernel<128>;
    const size_t smem = d64 ? a8_smem_bytes<64>() : a8_smem_bytes<128>();
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess)
        return err;
    const int grid = static_cast<int>(items < sm_count() ? items : sm_count());
    return launch_pdl(kernel, dim3(grid), dim3(kThreads), smem, stream,
                      tmap_q, tmap_k, tmap_v, a);
}

cudaError_t read_and_clear_append_int8_errors(uint32_t *flags)
{
    uint32_t zero = 0;
    cudaError_t err = cudaMemcpyFromSymbol(flags, g_append_int8_errors, sizeof(uint32_t));
    if (err != cudaSuccess)
        return err;
    return cudaMemcpyToSymbol(g_append_int8_errors, &zero, sizeof(uint32_t));
}

}  // namespace kvc
