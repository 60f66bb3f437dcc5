// kvc_append_tc.cu -- causal chunked prefill over a paged cached prefix on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// What it computes: Quail "KV", "KV rewind" and "Prefix sharing"; TileInfer.jl "KV cache",
// "Prefix reuse in chat".  New token i of a sequence (ctx positions, q_len new) sits at
// position ctx - q_len + i and attends to positions 0 .. ctx - q_len + i, read in place from
// the pages its block table lists.
//
// Tiling: the rows of one (sequence, kv head) are its (new token, query head of the group)
// pairs, token-major, in tiles of 128 (the tcgen05 M).  A work item is a pair of consecutive
// tiles of one (sequence, kv head); both tiles attend over the same pages, so every K or V
// stage loaded for the item feeds two tiles.  The kernel is persistent: one CTA per SM walks
// items c, c + grid, ... and its roles run ahead across item boundaries:
//   warp 0      TMA, K and V: 128-position stages (one box per page and 64-column half,
//               128-byte swizzle, the boxes of a stage issued by parallel lanes), K(b) and V(b)
//               in separate slots of one ring filled in the order K(0), K(1), V(0), K(2), V(1),
//               ..., so V(b) lands next to K(b + 1), about when PV(b) needs it, and a K slot is
//               refilled as soon as both tiles' S = Q K^T products have read it;
//   warp 1      allocates TMEM (512 columns) and issues, from one thread and in a fixed order,
//               S_w = Q_w K(b)^T (M 128, N 128, K head_dim) and O_w += P_w V(b) (M 128,
//               N head_dim, K 128, P read from TMEM) for the tiles w.  tcgen05.mma issue
//               blocks while the tensor pipe is busy, so this warp does nothing else; products
//               of one thread run in issue order, so S_w(b + 1) is issued right behind the PV
//               product that reads P_w(b) from the same columns.  Before the last PV of an
//               item it zeroes the V rows between the last visible position and the next
//               multiple of 16, so NaN or Inf left in unused slots never meets a zero
//               probability inside the tensor core;
//   warp 2      TMA, the item's query tiles (one buffer per tile, refilled once that tile's
//               last S product of the item is done);
//   warps 3-6   softmax of tile 0, warps 7-10 softmax of tile 1: thread r owns row r (TMEM
//               lane r; warp w reaches lanes 32 (w % 4) ..): reads its S row, applies the
//               scale and the causal limit, keeps a running max / sum, writes P (bf16 pairs)
//               over the first half of the S columns, and at the end of the item writes O / l.
//   (kvc_append_store) warp 2 also writes the chunk's rows from the ring slots they landed in
//               (read from k_new / v_new there) to the pools, and releases each slot on a
//               barrier of its own that the K/V producer waits for as well.
// The running max is updated lazily: O is rescaled (in TMEM) only when a row's max grows by
// more than 2^8.  The result is exact either way; probabilities are then at most 2^8 before
// normalisation.  Barrier phases follow counters kept identically by every role (items, ring
// slots, and each tile's blocks and items), so they line up across items.
#include <math.h>

#include "kvc_append_items.cuh"
#include "kvc_device.cuh"
#include "kvc_launch.h"

namespace kvc {

namespace {

__device__ uint32_t g_append_tc_errors;

using append::Item;
using append::kBN;   // positions per K or V stage (the N of S = Q K^T)
using append::kM;    // rows per tile
using append::seq_of;
using append::Walker;
constexpr int kRoleWarps = 3;     // K/V loads, MMA issue, query loads
constexpr int kSoftmaxWarps = 8;  // two groups of four
constexpr int kThreads = (kRoleWarps + kSoftmaxWarps) * 32;
constexpr int kMaxStages = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;

template <int D>
struct TcGeom {
    static constexpr int kHalves = D / 64;
    static constexpr int kQBytes = kHalves * kM * 128;       // one query tile
    static constexpr int kStageBytes = kHalves * kBN * 128;  // K or V of 128 positions
    static constexpr int kStages = D == 128 ? 5 : 8;
    static constexpr int kOffStages = 2 * kQBytes;           // Q: [tile]
    static constexpr int kOffBar = kOffStages + kStages * kStageBytes;
    static constexpr size_t kSmemBytes = kOffBar + 512;      // base is 1024-aligned
    // TMEM, per tile w at w * 256: O [0, D), S [D, D + 128); P overwrites S [D, D + 64).
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = D;
    static_assert(D + kBN <= 256, "TMEM layout");
    static_assert(kStages <= kMaxStages, "ring barriers");
    static_assert(kSmemBytes <= 232448, "shared memory");
};

struct Args {
    void *out;
    int out_f32;
    const int32_t *block_table;
    int bt_stride;
    const int32_t *q_indptr;
    const int32_t *context_lens;
    int kv_heads, q_heads, group, page_size, pairs_per_seq, num_items;
    float scale_log2;
    int hnd;   // HND pools: half boxes addressed by (offset, page * kv_heads + kv head)
    // Fused store (kvc_append_store): the chunk's pages are read from k_new / v_new and written
    // to the pools by this kernel, except the tokens that share a page with cached positions
    // (stored before the launch).
    int fused;
    uint8_t *k_pool_w, *v_pool_w;   // the pools, for rows of a partly filled last page
    int num_pages;                  // their pages (a page id outside them is skipped)
    uint32_t *err;                  // the caller's device error word, or null (this file's own)
};

enum BarIndex : int {
    kBarKvFull = 0,                         // [ring slot]
    kBarKvEmpty = kBarKvFull + kMaxStages,  // [ring slot], one MMA commit
    kBarQFull = kBarKvEmpty + kMaxStages,   // [tile]
    kBarQEmpty = kBarQFull + 2,             // [tile], one MMA commit after its last S product
    kBarSFull = kBarQEmpty + 2,             // [tile]
    kBarPFull = kBarSFull + 2,              // [tile], 128 arrivals
    kBarPvDone = kBarPFull + 2,             // [tile], once per item
    kBarDrain = kBarPvDone + 2,
    kBarKvStored = kBarDrain + 1,           // [ring slot], fused store: its pages written
    kBarCount = kBarKvStored + kMaxStages
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    paged_append_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                           const __grid_constant__ CUtensorMap tmap_k,
                           const __grid_constant__ CUtensorMap tmap_v,
                           const __grid_constant__ CUtensorMap tmap_kn,
                           const __grid_constant__ CUtensorMap tmap_vn, const Args a)
{
    pdl_wait();
    pdl_trigger();
    uint32_t *const err_word = a.err ? a.err : &g_append_tc_errors;
    using Geom = TcGeom<D>;
    constexpr int kHalves = D / 64;
    constexpr int kStages = Geom::kStages;

    // The swizzled tiles need a 1024-byte-aligned base; the dynamic shared window of a kernel
    // with no static shared memory starts there, which is checked rather than padded for.
    extern __shared__ __align__(1024) uint8_t smem[];
    if ((smem_addr(smem) & 1023u) != 0) {
        if (threadIdx.x == 0)
            atomicOr(err_word, kErrSmemAlign);
        return;
    }
    uint8_t *sStages = smem + Geom::kOffStages;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Geom::kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kBarCount);
    auto q_tile = [&](int tile) { return smem + tile * Geom::kQBytes; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.group;
    const int P = a.page_size;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kBarCount; ++i)
            mbar_init(&bars[i], (i == kBarPFull || i == kBarPFull + 1) ? 128u : 1u);
        fence_mbar_init();
    }
    if (warp == 1)
        tmem_alloc(tmem_slot, Geom::kTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        // ------------------------------ K / V loads --------------------------------------
        if (lane == 0) {
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
        }
        const uint64_t policy = l2_policy_evict_first();
        Walker w;
        w.start(a, err_word);
        // block-table entries 0 .. 31 of the current item's sequence, one per lane, requested
        // one item ahead like the item metadata
        auto bt_head = [&](int idx) {
            return (idx < a.num_items && lane < a.bt_stride)
                       ? a.block_table[static_cast<size_t>(seq_of(a, idx)) * a.bt_stride + lane]
                       : 0;
        };
        int head_it = w.done ? -1 : w.it;
        int head_page = w.done ? 0 : bt_head(w.it);
        int n = 0;   // ring slots filled so far
        while (ok && !w.done) {
            const Item &x = w.x;
            const int32_t *bt_row = a.block_table + static_cast<size_t>(x.s) * a.bt_stride;
            const int n_pages = (x.n_keys + P - 1) / P;
            int cached_base = 0;
            int cached_page = (head_it == w.it) ? head_page : bt_head(w.it);
            head_it = w.it + static_cast<int>(gridDim.x);   // the next index, if not skipped
            head_page = bt_head(head_it);
            const int nb = x.n_blocks;
            const int base = x.ctx - x.q_len;   // position of the chunk's first token
            const int first_new = base > 0 ? (base + P - 1) / P : 0;
            for (int j = 0; j < 2 * nb; ++j, ++n) {
                // Fill order K(0), K(1), V(0), K(2), V(1), ..., V(nb - 1): K runs one block
                // ahead, so V(b) lands about when PV(b) needs it, next to K(b + 1).
                const bool is_k = j == 0 || (j < 2 * nb - 1 && (j & 1));
                const int b = is_k ? (j + 1) / 2 : (j == 2 * nb - 1 ? nb - 1 : j / 2 - 1);
                const int key0 = b * kBN;
                const int np = (min(kBN, x.n_keys - key0) + P - 1) / P;
                {
                    const int st = n % kStages;
                    if (n >= kStages &&
                        (!__all_sync(0xffffffffu, mbar_wait(&bars[kBarKvEmpty + st],
                                                            ((n / kStages) - 1) & 1)) ||
                         (a.fused && !__all_sync(0xffffffffu,
                                                 mbar_wait(&bars[kBarKvStored + st],
                                                           ((n / kStages) - 1) & 1))))) {
                        ok = false;
                        break;
                    }
                    if (lane == 0)
                        mbar_arrive_expect_tx(&bars[kBarKvFull + st],
                                              static_cast<uint32_t>(np * P * D * 2));
                    __syncwarp();
                    uint8_t *dst = sStages + st * Geom::kStageBytes;
                    const CUtensorMap *map = is_k ? &tmap_k : &tmap_v;
                    const int lp0 = key0 / P;   // first page of the block
                    if (lp0 < cached_base || lp0 + np > cached_base + 32) {
                        cached_base = lp0;
                        cached_page = (lp0 + lane < n_pages) ? bt_row[lp0 + lane] : 0;
                    }
                    // Lane i * kHalves + h issues the box of page i, column half h: boxes issued
                    // by one thread one after another run at a fraction of the TMA rate that
                    // lanes issuing together reach for these small boxes.
                    const int i = lane / kHalves;
                    const int h = lane % kHalves;
                    const int page =
                        __shfl_sync(0xffffffffu, cached_page, (lp0 - cached_base + i) & 31);
                    // NHD maps {head_dim, kv head, slot}; HND maps {head_dim, offset, block}.
                    // Fused store: a page that holds only the chunk's tokens comes from
                    // k_new / v_new ({head_dim, kv head, token}), its first token at
                    // tok0 + lp * P - (ctx - q_len).
                    const int lp = lp0 + i;
                    if (i < np && a.fused && lp >= first_new)
                        tma_load_3d(dst + h * kBN * 128 + i * P * 128, is_k ? &tmap_kn : &tmap_vn,
                                    h * 64, x.kvh, x.tok0 + lp * P - base, &bars[kBarKvFull + st],
                                    policy);
                    else if (i < np)
                        tma_load_3d(dst + h * kBN * 128 + i * P * 128, map, h * 64,
                                    a.hnd ? 0 : x.kvh, a.hnd ? page * a.kv_heads + x.kvh : page * P,
                                    &bars[kBarKvFull + st], policy);
                }
            }
            if (!ok)
                break;
            w.next(a, err_word);
        }
        if (!ok && lane == 0) {
            atomicOr(err_word, kErrAppendTcWait);
            // let every copy in flight land before the CTA can exit
            for (int m = max(0, n - kStages); m < n; ++m)
                if (!mbar_wait(&bars[kBarKvFull + m % kStages], (m / kStages) & 1))
                    atomicOr(err_word, kErrDrainWait);
        }
    } else if (warp == 2) {
        // ------------------------------ query loads (and the fused store) -----------------
        if (lane == 0)
            prefetch_tensormap(&tmap_q);
        Walker w;
        w.start(a, err_word);
        int qi[2] = {0, 0};   // items whose query tile t was requested
        int n = 0;
        while (ok && !w.done) {
            const Item &x = w.x;
            // Tile t of the next item loads as soon as tile t of this one has had its last S
            // product, so tile 0 can start before tile 1 is free.  Lane h loads column half h
            // of the tile's 128 / G tokens x G heads of this kv head, token-major.
            for (int t = 0; t < (x.has_b ? 2 : 1); ++t) {
                if (qi[t] > 0 &&
                    !__all_sync(0xffffffffu,
                                mbar_wait(&bars[kBarQEmpty + t], (qi[t] - 1) & 1))) {
                    ok = false;
                    break;
                }
                if (lane == 0)
                    mbar_arrive_expect_tx(&bars[kBarQFull + t],
                                          static_cast<uint32_t>(Geom::kQBytes));
                __syncwarp();
                if (lane < kHalves)
                    tma_load_4d(q_tile(t) + lane * kM * 128, &tmap_q, lane * 64, 0, x.kvh,
                                x.tok0 + (x.row_begin + t * kM) / G, &bars[kBarQFull + t]);
                ++qi[t];
            }
            if (!ok)
                break;
            if (a.fused) {
                // Fused store: write the chunk's positions that this tile pair sees and no
                // earlier pair of its (sequence, kv head) saw, [p_lo, p_hi), row by row from
                // the ring slots they landed in (16-byte loads and stores; measured as fast as
                // TMA stores of whole pages, and a slot is free once its rows are in registers).
                // Rows at or past p_hi = n_keys may be zeroed by the MMA warp for the last PV
                // product; they are never read here.  Positions in the page of the chunk's first
                // token that also holds cached ones were stored before the launch.  Every slot
                // gets its arrival on kBarKvStored once it has landed: a parity wait cannot
                // tell a phase from the one two later, so this warp must not run two phases of
                // kBarKvStored ahead of the producer's waits.
                const int nb = x.n_blocks;
                const int base = x.ctx - x.q_len;
                const int first_new = base > 0 ? (base + P - 1) / P : 0;
                int p_lo = first_new * P;
                if (x.tp > 0)
                    p_lo = max(p_lo, min(x.ctx, base + (x.row_begin - 1) / G + 1));
                const int p_hi = x.n_keys;
                const int32_t *bt_row = a.block_table + static_cast<size_t>(x.s) * a.bt_stride;
                for (int j = 0; j < 2 * nb; ++j, ++n) {
                    const bool is_k = j == 0 || (j < 2 * nb - 1 && (j & 1));
                    const int b = is_k ? (j + 1) / 2 : (j == 2 * nb - 1 ? nb - 1 : j / 2 - 1);
                    const int st = n % kStages;
                    const int lp0 = b * kBN / P;
                    const int np = (min(kBN, x.n_keys - b * kBN) + P - 1) / P;
                    const int s_lo = max(lp0, p_lo / P);   // pages of the block to write
                    const int s_hi = min(lp0 + np, (p_hi + P - 1) / P);
                    // (a context past its block-table row: the whole chunk was stored by
                    // the boundary kernel at the slots the row covers, as slot mapping +
                    // store would; nothing is written here)
                    const bool write = !x.over && p_lo < p_hi && s_lo < s_hi;
                    const int my_page = (write && s_lo + lane < s_hi) ? bt_row[s_lo + lane] : 0;
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(&bars[kBarKvFull + st], (n / kStages) & 1))) {
                        ok = false;
                        break;
                    }
                    if (write) {
                        const uint8_t *stage = sStages + st * Geom::kStageBytes;
                        uint8_t *pool = is_k ? a.k_pool_w : a.v_pool_w;
                        for (int lp = s_lo; lp < s_hi; ++lp) {
                            const int page = __shfl_sync(0xffffffffu, my_page, lp - s_lo);
                            if (page < 0 || page >= a.num_pages) {   // outside the pool: skip, flag
                                if (lane == 0)
                                    atomicOr(err_word, kErrSlotRange);
                                continue;
                            }
                            const int i = lp - lp0;
                            const int r_lo = max(p_lo - lp * P, 0);
                            const int r_hi = min(p_hi - lp * P, P);
                            // rows r_lo .. r_hi - 1; 16-byte chunk c of row r sits at chunk
                            // (c % 8) ^ (r % 8) of its 128-byte line
                            for (int idx = lane; idx < (r_hi - r_lo) * (D / 8); idx += 32) {
                                const int c = idx % (D / 8);
                                const int r = r_lo + idx / (D / 8);
                                const uint4 v = *reinterpret_cast<const uint4 *>(
                                    stage + (c >> 3) * kBN * 128 + (i * P + r) * 128 +
                                    (((c & 7) ^ (r & 7)) << 4));
                                const size_t row =
                                    a.hnd ? (static_cast<size_t>(page) * a.kv_heads + x.kvh) * P +
                                                r
                                          : (static_cast<size_t>(page) * P + r) * a.kv_heads +
                                                x.kvh;
                                *reinterpret_cast<uint4 *>(pool + row * (D * 2) + c * 16) = v;
                            }
                        }
                        __syncwarp();
                    }
                    if (lane == 0)
                        mbar_arrive(&bars[kBarKvStored + st]);
                }
                if (!ok)
                    break;
            }
            if (!ok)
                break;
            w.next(a, err_word);
        }
        if (!ok && lane == 0) {
            atomicOr(err_word, kErrAppendTcWait);
            // the last requests may still be in flight
            for (int t = 0; t < 2; ++t)
                if (qi[t] > 0 && !mbar_wait(&bars[kBarQFull + t], (qi[t] - 1) & 1))
                    atomicOr(err_word, kErrDrainWait);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issue ----------------------------------------
        constexpr uint32_t kIdescPV = umma_idesc_bf16(kM, D, 1);
        const uint32_t stage_addr = smem_addr(sStages);
        auto stage_of = [&](int n) { return stage_addr + (n % kStages) * Geom::kStageBytes; };
        auto wait_slot = [&](int n) {
            return __all_sync(0xffffffffu,
                              mbar_wait(&bars[kBarKvFull + n % kStages], (n / kStages) & 1));
        };
        // S_t = Q_t K^T over n_cols positions (a multiple of 16)
        auto issue_qk = [&](int t, uint32_t k_addr, int n_cols) {
            const uint32_t idesc = umma_idesc_bf16(kM, n_cols, 0);
            const uint32_t q_addr = smem_addr(q_tile(t));
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint64_t da =
                    umma_desc_sw128(q_addr + (k >> 2) * kM * 128 + (k & 3) * 32, 16, 1024);
                const uint64_t db =
                    umma_desc_sw128(k_addr + (k >> 2) * kBN * 128 + (k & 3) * 32, 16, 1024);
                umma_bf16_ss(tmem + t * 256 + Geom::kColS, da, db, idesc, k > 0 ? 1u : 0u);
            }
        };
        // O_t (+)= P_t V over k_steps x 16 positions
        auto issue_pv = [&](int t, uint32_t v_addr, int k_steps, bool first) {
            for (int k = 0; k < k_steps; ++k) {
                const uint64_t db = umma_desc_sw128(v_addr + k * 16 * 128, kBN * 128, 1024);
                umma_bf16_ts(tmem + t * 256, tmem + t * 256 + Geom::kColS + k * 8, db, kIdescPV,
                             (!first || k > 0) ? 1u : 0u);
            }
        };
        Walker w;
        w.start(a, err_word);
        int n0 = 0;             // ring index of the item's first slot
        int qi[2] = {0, 0};     // items of tile 0 / tile 1
        int tb[2] = {0, 0};     // blocks of tile 0 / tile 1
        while (ok && !w.done) {
            const Item &x = w.x;
            const int nt = x.has_b ? 2 : 1;
            const int nb = x.n_blocks;
            const int last_valid = x.n_keys - (nb - 1) * kBN;   // positions in the last block
            const int last_cols = (last_valid + 15) & ~15;
            // ring indices in the producer's fill order K(0), K(1), V(0), K(2), V(1), ...
            auto k_slot = [&](int b) { return n0 + (b == 0 ? 0 : 2 * b - 1); };
            auto v_slot = [&](int b) { return n0 + (b == nb - 1 ? 2 * nb - 1 : 2 * b + 2); };
            if (!wait_slot(k_slot(0))) {
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
                    issue_qk(t, stage_of(k_slot(0)), nb == 1 ? last_cols : kBN);
                    umma_commit(&bars[kBarSFull + t]);
                    if (nb == 1)
                        umma_commit(&bars[kBarQEmpty + t]);
                }
                __syncwarp();
            }
            if (!ok)
                break;
            if (lane == 0)
                umma_commit(&bars[kBarKvEmpty + k_slot(0) % kStages]);
            __syncwarp();
            for (int b = 0; b < nb && ok; ++b) {
                const bool last = b + 1 == nb;
                const int vn = v_slot(b);
                if (!wait_slot(vn)) {
                    ok = false;
                    break;
                }
                if (last && last_valid < last_cols) {
                    // V rows last_valid .. last_cols - 1 of every column half
                    uint8_t *vt = sStages + (vn % kStages) * Geom::kStageBytes;
                    const int rows_to_zero = last_cols - last_valid;
                    for (int idx = lane; idx < rows_to_zero * kHalves * 8; idx += 32) {
                        const int chunk = idx & 7;
                        const int rest = idx >> 3;
                        const int h = rest % kHalves;
                        const int r = last_valid + rest / kHalves;
                        *reinterpret_cast<uint4 *>(vt + h * kBN * 128 + r * 128 + chunk * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                const int kn = last ? 0 : k_slot(b + 1);
                for (int t = 0; t < nt; ++t) {
                    if (!__all_sync(0xffffffffu, mbar_wait(&bars[kBarPFull + t], tb[t] & 1))) {
                        ok = false;
                        break;
                    }
                    ++tb[t];
                    tc_fence_after_sync();
                    if (lane == 0) {
                        issue_pv(t, stage_of(vn), last ? last_cols / 16 : kBN / 16, b == 0);
                        if (last)
                            umma_commit(&bars[kBarPvDone + t]);
                    }
                    __syncwarp();
                    if (last)
                        continue;
                    // K(b + 1) is waited for only once PV(b) of tile 0 is on its way
                    if (t == 0 && !wait_slot(kn)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    if (lane == 0) {
                        issue_qk(t, stage_of(kn), b + 2 == nb ? last_cols : kBN);
                        umma_commit(&bars[kBarSFull + t]);
                        if (b + 2 == nb)
                            umma_commit(&bars[kBarQEmpty + t]);
                    }
                    __syncwarp();
                }
                if (!ok)
                    break;
                if (lane == 0) {
                    umma_commit(&bars[kBarKvEmpty + vn % kStages]);
                    if (!last)
                        umma_commit(&bars[kBarKvEmpty + kn % kStages]);
                }
                __syncwarp();
            }
            if (!ok)
                break;
            for (int t = 0; t < nt; ++t)
                ++qi[t];
            n0 += 2 * nb;
            w.next(a, err_word);
        }
        if (!ok && lane == 0)
            atomicOr(err_word, kErrAppendTcWait);
        // Every MMA this thread issued must be complete before TMEM is released.
        if (lane == 0) {
            umma_commit(&bars[kBarDrain]);
            if (!mbar_wait(&bars[kBarDrain], 0))
                atomicOr(err_word, kErrDrainWait);
        }
        __syncwarp();
    } else {
        // ------------------------------ softmax + epilogue -------------------------------
        const int t = (warp - kRoleWarps) >> 2;      // tile
        const int quad = warp & 3;                   // TMEM lanes 32 quad ..
        const int row = quad * 32 + lane;            // row of the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tmem_o = tmem + t * 256 + lane_off;
        const uint32_t tmem_s = tmem + t * 256 + Geom::kColS + lane_off;
        const float sl2 = a.scale_log2;
        Walker w;
        w.start(a, err_word);
        int tb = 0;   // blocks of this tile so far
        int ti = 0;   // items of this tile so far
        for (; ok && !w.done; w.next(a, err_word)) {
            const Item &x = w.x;
            if (t == 1 && !x.has_b)
                continue;
            const int row_begin = x.row_begin + t * kM;
            const int gr = row_begin + row;
            const bool valid = gr < x.rows;
            const int tok = gr / G;
            const int lim = valid ? x.ctx - x.q_len + tok : -1;   // last visible position
            const bool warp_valid = __any_sync(0xffffffffu, valid);
            float m_used = -INFINITY;
            float l_sum = 0.0f;
            for (int b = 0; b < x.n_blocks; ++b, ++tb) {
                if (!__all_sync(0xffffffffu, mbar_wait(&bars[kBarSFull + t], tb & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const int key0 = b * kBN;
                // positions of this block the row may see: columns 0 .. n_vis - 1
                const int n_vis = min(max(lim - key0 + 1, 0), kBN);
                float alpha = 1.0f;
                bool moved = false;
                if (warp_valid) {
                    // pass 1: the row max; masked columns are set to -inf in TMEM as well, so
                    // the exponent pass below needs no mask
                    float xs[4][32];
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        tmem_ld32(tmem_s + 32 * c, xs[c]);
                    tmem_wait_ld();
                    float mx = -INFINITY;
                    if (__all_sync(0xffffffffu, n_vis == kBN)) {
#pragma unroll
                        for (int j = 0; j < kBN; j += 2)
                            mx = fmax3(mx, xs[j >> 5][j & 31], xs[j >> 5][(j & 31) + 1]);
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (32 * c + j >= n_vis)
                                    xs[c][j] = -INFINITY;
#pragma unroll
                            for (int j = 0; j < 32; j += 2)
                                mx = fmax3(mx, xs[c][j], xs[c][j + 1]);
                            tmem_st32(tmem_s + 32 * c, xs[c]);
                        }
                        tmem_wait_st();
                    }
                    const float mb = mx * sl2;   // base-2 scaled row max of this block
                    if (mb > m_used + kRescaleLog2) {
                        alpha = (m_used == -INFINITY) ? 0.0f : fast_exp2(m_used - mb);
                        m_used = mb;
                        moved = true;
                    }
                }
                // O holds every earlier PV product (S(b) was committed after them): rescale
                // it in place when the max moved.
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
                // pass 2, 32 columns at a time (a short loop body keeps the instruction
                // footprint small), in paired fp32 arithmetic: p = 2^(s * scale * log2(e) - m)
                // on MUFU (measured: moving a share of the exponentials to an FMA-pipe
                // polynomial costs more issue slots than it saves); the bf16 pairs of chunk c go
                // to S columns [16 c, 16 c + 16), which hold only chunks already read; the sum
                // takes the rounded bf16 values.
                const float neg_mu = (m_used == -INFINITY) ? 0.0f : -m_used;
                const uint64_t sl2x2 = f2_pack(sl2, sl2);
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
                        for (int j = 0; j < 16; ++j) {
                            float e0, e1;
                            f2_unpack(f2_fma(f2_pack(v[2 * j], v[2 * j + 1]), sl2x2, nm2), e0, e1);
                            pk[j] = pack_bf16x2(fast_exp2(e0), fast_exp2(e1));
                            psum2 = f2_add(psum2, f2_pack(__uint_as_float(pk[j] << 16),
                                                          __uint_as_float(pk[j] & 0xFFFF0000u)));
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j)   // a warp of padding rows: P = 0
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
            atomicOr(err_word, kErrAppendTcWait);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, Geom::kTmemCols);
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

template <int D>
cudaError_t launch_t(const AppendLaunch &l, const CUtensorMap &tq, const CUtensorMap &tk,
                     const CUtensorMap &tv, const CUtensorMap &tkn, const CUtensorMap &tvn,
                     cudaStream_t stream)
{
    Args a;
    a.out = l.out;
    a.out_f32 = l.out_f32;
    a.block_table = l.block_table;
    a.bt_stride = l.bt_stride;
    a.q_indptr = l.q_indptr;
    a.context_lens = l.context_lens;
    a.kv_heads = l.kv_heads;
    a.q_heads = l.q_heads;
    a.group = l.q_heads / l.kv_heads;
    a.page_size = l.page_size;
    a.hnd = l.hnd ? 1 : 0;
    a.fused = l.fused ? 1 : 0;
    a.k_pool_w = static_cast<uint8_t *>(l.k_pool_w);
    a.v_pool_w = static_cast<uint8_t *>(l.v_pool_w);
    a.num_pages = l.num_pages;
    a.err = current_error_word();
    const int tiles = (l.max_q_len * a.group + kM - 1) / kM;
    a.pairs_per_seq = (tiles + 1) / 2;
    const long long items = static_cast<long long>(a.pairs_per_seq) * l.kv_heads * l.num_seqs;
    if (items > 0x7FFFFFFFLL)
        return cudaErrorInvalidValue;
    a.num_items = static_cast<int>(items);
    a.scale_log2 = l.scale * kLog2e;
    const size_t smem = TcGeom<D>::kSmemBytes;
    auto kernel = paged_append_tc_kernel<D>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess)
        return err;
    const int grid = static_cast<int>(items < sm_count() ? items : sm_count());
    return launch_pdl(kernel, dim3(grid), dim3(kThreads), smem, stream, tq, tk, tv, tkn, tvn, a);
}

}  // namespace

cudaError_t launch_append_tc(const AppendLaunch &l, const CUtensorMap &tmap_q,
                             const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                             cudaStream_t stream, const CUtensorMap *tmap_kn,
                             const CUtensorMap *tmap_vn)
{
    if (l.num_seqs == 0 || l.num_tokens == 0 || l.max_q_len == 0)
        return cudaSuccess;
    if (l.fused && (tmap_kn == nullptr || tmap_vn == nullptr))
        return cudaErrorInvalidValue;
    const CUtensorMap &kn = tmap_kn ? *tmap_kn : tmap_k;   // unused unless fused
    const CUtensorMap &vn = tmap_vn ? *tmap_vn : tmap_v;
    return l.head_dim == 128 ? launch_t<128>(l, tmap_q, tmap_k, tmap_v, kn, vn, stream)
                             : launch_t<64>(l, tmap_q, tmap_k, tmap_v, kn, vn, stream);
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
