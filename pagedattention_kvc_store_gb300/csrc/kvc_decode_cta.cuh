// kvc_decode_cta.cuh -- the work of one decode CTA: one (split, kv head, sequence) of paged
// decode attention, "KV Cache Management and PagedAttention", "Compute attention over
// scattered KV".  kvc_decode.cu launches it as paged_decode_kernel (its design is described
// there); the shared-prefix decode runs it for the members' suffixes inside the same grid as
// its prefix CTAs (kvc_grouped.cu).
#pragma once

#include <math.h>

#include "kvc_device.cuh"
#include "kvc_launch.h"

namespace kvc {
namespace dec {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 3;
constexpr int kKeysPerWarp = kStageKeys / kConsumerWarps;   // 16
constexpr int kMaxGroup = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

static_assert(kKeysPerWarp == 16, "each consumer warp covers one 16-position MMA k-step");

template <int D>
struct DecodeGeom {
    static constexpr int kTileBytes = kStageKeys * D * 2;   // K (or V) of one stage
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kRingBytes = kStages * kStageBytes;
    // after the ring: full[kStages], empty[kStages] mbarriers
    static constexpr int kBarrierBytes = 2 * kStages * 8;
    static constexpr int kCombineBytes =   // o rows, m, l per warp; weights per row
        kConsumerWarps * kMaxGroup * (D + 8) * 4 + 3 * kConsumerWarps * kMaxGroup * 4;
    static_assert(kCombineBytes <= kRingBytes, "combine area aliases the ring");
    static constexpr size_t kSmemBytes = 1024 /* alignment slack */ + kRingBytes + kBarrierBytes;
};

struct Args {
    const __nv_bfloat16 *q;
    void *out;
    int out_f32;
    float *part_o;
    float *part_lse;
    const int32_t *block_table;
    int bt_stride;
    const int32_t *context_lens;
    const int32_t *key_start;   // optional [S]: positions below it are another kernel's
    int q_heads, kv_heads, group, page_size;
    int chunk, n_split;
    int split_base, split_stride;   // partial j of this launch is split split_base + j of
                                    // split_stride per row
    float scale_log2;
    int hnd;                        // HND pools: page boxes addressed by (page, kv head) block
    // Fused store (kvc_decode_store): the new token of every sequence, [S][Hkv][D], written
    // into the pools (num_slots slots) by the CTA whose chunk ends at the newest position,
    // before that CTA's copy of the page; null otherwise.
    const uint4 *k_new, *v_new;
    uint4 *k_pool, *v_pool;
    int num_slots;
    uint32_t *err;   // the caller's device error word, or null (the kernel's own word)
};

// Kernel arguments from the host-side launch description.
inline Args make_args(const DecodeLaunch &l)
{
    Args a;
    a.q = static_cast<const __nv_bfloat16 *>(l.q);
    a.out = l.out;
    a.out_f32 = l.out_f32;
    a.part_o = l.part_o;
    a.part_lse = l.part_lse;
    a.block_table = l.block_table;
    a.bt_stride = l.bt_stride;
    a.context_lens = l.context_lens;
    a.key_start = l.key_start;
    a.q_heads = l.q_heads;
    a.kv_heads = l.kv_heads;
    a.hnd = l.hnd ? 1 : 0;
    a.group = l.q_heads / l.kv_heads;
    a.page_size = l.page_size;
    a.chunk = l.chunk;
    a.n_split = l.n_split;
    a.split_base = l.split_base;
    a.split_stride = l.split_stride > 0 ? l.split_stride : l.n_split;
    a.scale_log2 = l.scale * kLog2e;
    a.k_new = static_cast<const uint4 *>(l.k_new);
    a.v_new = static_cast<const uint4 *>(l.v_new);
    a.k_pool = static_cast<uint4 *>(l.k_pool_w);
    a.v_pool = static_cast<uint4 *>(l.v_pool_w);
    a.num_slots = l.num_slots;
    a.err = current_error_word();
    return a;
}

// One CTA (kThreads threads, DecodeGeom<D>::kSmemBytes of dynamic shared memory, `smem`
// 1024-byte aligned) on chunk `split` of kv head `kvh` of sequence `s`; device-side failures
// are or-ed into *errors.
template <int D, bool SPLIT>
__device__ __forceinline__ void decode_cta(const CUtensorMap *tmap_k, const CUtensorMap *tmap_v,
                                           const Args &a, const int split, const int kvh,
                                           const int s, uint8_t *smem, uint32_t *errors)
{
    using Geom = DecodeGeom<D>;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Geom::kRingBytes);
    uint64_t *empty = full + kStages;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.group;
    const int P = a.page_size;
    const int k_first = a.key_start ? a.key_start[s] : 0;   // a multiple of page_size
    const int k_begin = k_first + split * a.chunk;
    // The producer's first 32 page ids are requested together with the context length (the
    // chunk's first page does not depend on it), one memory round trip less before the first
    // TMA copy; entries past the sequence's pages are read but never used.
    int pre_page = 0;
    if (warp == kConsumerWarps && k_begin / P + lane < a.bt_stride)
        pre_page = a.block_table[static_cast<size_t>(s) * a.bt_stride + k_begin / P + lane];
    // Fused store: the producer's lanes fetch the sequence's new K / V row for this kv head
    // (16 bytes each) together with the context length; only the CTA whose chunk ends at the
    // newest position writes it.
    constexpr int kRowChunks = D / 8;
    uint4 k_row_new = make_uint4(0u, 0u, 0u, 0u), v_row_new = k_row_new;
    if (a.k_new != nullptr && warp == kConsumerWarps && lane < kRowChunks) {
        const size_t src = (static_cast<size_t>(s) * a.kv_heads + kvh) * kRowChunks + lane;
        k_row_new = load_streaming(a.k_new + src);
        v_row_new = load_streaming(a.v_new + src);
    }
    int ctx = a.context_lens[s];
    bool store_new = a.k_new != nullptr && ctx >= 1;
    if (ctx > a.bt_stride * a.page_size) {   // the block-table row cannot hold it
        if (threadIdx.x == 0 && split == 0)
            atomicOr(errors, kErrContextRange);
        ctx = a.bt_stride * a.page_size;
        store_new = false;                    // no slot for the new token: stored nowhere
    }
    const int k_end = min(ctx, k_begin + a.chunk);
    const size_t row0 = static_cast<size_t>(s) * a.q_heads + static_cast<size_t>(kvh) * G;

    if (k_begin >= k_end) {
        // This chunk holds no position of the sequence.
        if (SPLIT) {
            if (threadIdx.x < G)
                a.part_lse[(row0 + threadIdx.x) * a.split_stride + a.split_base + split] =
                    -INFINITY;
        } else {
            for (int i = threadIdx.x; i < G * D; i += blockDim.x)
                store_out(a.out, a.out_f32, row0 * D + i, 0.0f);
        }
        return;
    }

    const int n_blocks = (k_end - k_begin + kStageKeys - 1) / kStageKeys;
    const int first_page = k_begin / P;
    const int n_pages = (k_end - k_begin + P - 1) / P;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------ TMA producer (whole warp) -------------------------------
        // Page ids are read 32 at a time by the warp's lanes and handed to lane 0, which
        // issues the copies.
        const int32_t *bt_row =
            a.block_table + static_cast<size_t>(s) * a.bt_stride + first_page;
        if (lane == 0) {
            prefetch_tensormap(tmap_k);
            prefetch_tensormap(tmap_v);
        }
        const uint64_t policy = l2_policy_evict_first();
        const int shP = __ffs(P) - 1;   // page sizes are powers of two
        int cached_base = 0;
        int cached_page = pre_page;
        int issued = 0;
        bool ok = true;
        // this CTA writes the new token when its chunk ends at the newest position, in the
        // sequence's last page: before the last stage's copies read that page
        const bool writes_new = store_new && k_end == ctx;
        const int new_page = writes_new ? a.block_table[static_cast<size_t>(s) * a.bt_stride +
                                                        (ctx - 1) / P]
                                        : 0;
        for (int b = 0; b < n_blocks; ++b) {
            const int st = b % kStages;
            if (b >= kStages) {
                const bool waited = mbar_wait(&empty[st], ((b / kStages) - 1) & 1);
                if (!__all_sync(0xffffffffu, waited)) {
                    ok = false;
                    break;
                }
            }
            const int rel0 = b * kStageKeys;
            const int keys = min(kStageKeys, k_end - k_begin - rel0);
            const int np = (keys + P - 1) >> shP;
            if (lane == 0)
                mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>((np << shP) * D * 2 * 2));
            __syncwarp();
            uint8_t *kdst = smem + st * Geom::kStageBytes;
            uint8_t *vdst = kdst + Geom::kTileBytes;
            const int lp0 = rel0 >> shP;   // first page of the stage inside this chunk
            if (lp0 + np > cached_base + 32) {
                cached_base = lp0;
                cached_page = (lp0 + lane < n_pages) ? bt_row[lp0 + lane] : 0;
            }
            // Lane 2 i loads page i of K, lane 2 i + 1 page i of V: boxes issued together by
            // several lanes reach a much higher TMA rate than one thread issuing them in turn.
            const int i = lane >> 1;
            const int page = __shfl_sync(0xffffffffu, cached_page, (lp0 - cached_base + i) & 31);
            if (writes_new && b + 1 == n_blocks) {
                const int off_new = (ctx - 1) % P;
                const long long slot = static_cast<long long>(new_page) * P + off_new;
                if (new_page >= 0 && slot < a.num_slots) {
                    if (lane < kRowChunks) {
                        const size_t dst =
                            a.hnd ? ((static_cast<size_t>(new_page) * a.kv_heads + kvh) * P +
                                     off_new) * kRowChunks + lane
                                  : (static_cast<size_t>(slot) * a.kv_heads + kvh) * kRowChunks +
                                        lane;
                        a.k_pool[dst] = k_row_new;
                        a.v_pool[dst] = v_row_new;
                    }
                } else if (lane == 0) {
                    atomicOr(errors, kErrSlotRange);   // skipped, as kvc_store skips it
                }
                // the stores (generic proxy) before the copies (async proxy) that read them
                fence_proxy_async_global();
                __syncwarp();
                fence_proxy_async_global();
            }
            if (i < np) {
                const int off = i * P * D * 2;
                // NHD maps {64, slot, half, kv head}; HND maps {64, offset, half, block}
                const int c1 = a.hnd ? 0 : page << shP;
                const int c3 = a.hnd ? page * a.kv_heads + kvh : kvh;
                if (lane & 1)
                    tma_load_4d_hint(vdst + off, tmap_v, 0, c1, 0, c3, &full[st], policy);
                else
                    tma_load_4d_hint(kdst + off, tmap_k, 0, c1, 0, c3, &full[st], policy);
            }
            issued = b + 1;
        }
        if (!ok && lane == 0) {
            atomicOr(errors, kErrDecodeEmptyWait);
            // Let every copy already in flight land before the CTA can exit.
            for (int b = max(0, issued - kStages); b < issued; ++b)
                if (!mbar_wait(&full[b % kStages], (b / kStages) & 1))
                    atomicOr(errors, kErrDrainWait);
        }
        return;
    }

    // --------------------------------- consumers -----------------------------------------
    const int r = lane >> 2;          // fragment row = q head of the group (rows >= G: padding)
    const int cq = (lane & 3) * 2;    // fragment column pair
    uint32_t qa[D / 16][2];
    {
        const __nv_bfloat16 *qrow = a.q + (row0 + r) * D;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qa[kk][0] = r < G ? *reinterpret_cast<const uint32_t *>(qrow + kk * 16 + cq) : 0u;
            qa[kk][1] =
                r < G ? *reinterpret_cast<const uint32_t *>(qrow + kk * 16 + 8 + cq) : 0u;
        }
    }
    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
        o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
    float m_run = -INFINITY;   // running max (base-2 scaled scores) of row r
    float l_run = 0.0f;        // this thread's part of the running sum of row r

    // ldmatrix lane addresses (row/column inside this warp's 16 positions of a stage)
    const int k_row = warp * kKeysPerWarp + (lane & 7) + ((lane >> 4) << 3);
    const int k_col = ((lane >> 3) & 1) << 3;
    const int v_row = warp * kKeysPerWarp + (lane & 7) + (((lane >> 3) & 1) << 3);
    const int v_col = (lane >> 4) << 3;
    const int log2p = __ffs(P) - 1;
    const float sl2 = a.scale_log2;
    bool ok = true;

    for (int b = 0; b < n_blocks; ++b) {
        const int st = b % kStages;
        if (!mbar_wait(&full[st], (b / kStages) & 1)) {
            ok = false;
            break;
        }
        const uint32_t kbase = smem_addr(smem + st * Geom::kStageBytes);
        const uint32_t vbase = kbase + Geom::kTileBytes;
        const int n_valid = k_end - (k_begin + b * kStageKeys + warp * kKeysPerWarp);
        if (n_valid > 0) {
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kbase + page_tile_offset<D>(k_row, kk * 16 + k_col, log2p), b0, b1, b2,
                        b3);
                mma_bf16_16816(sc[0], qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
                mma_bf16_16816(sc[1], qa[kk][0], 0u, qa[kk][1], 0u, b2, b3);
            }
            float x[4] = {sc[0][0] * sl2, sc[0][1] * sl2, sc[1][0] * sl2, sc[1][1] * sl2};
            if (n_valid < kKeysPerWarp) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if ((i >> 1) * 8 + cq + (i & 1) >= n_valid)
                        x[i] = -INFINITY;
            }
            float mb = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
            const float m_new = fmaxf(m_run, mb);
            if (__any_sync(0xffffffffu, m_new > m_run)) {
                const float alpha = (m_run == -INFINITY) ? 0.0f : fast_exp2(m_run - m_new);
#pragma unroll
                for (int n = 0; n < D / 8; ++n) {
                    o[n][0] *= alpha;
                    o[n][1] *= alpha;
                }
                l_run *= alpha;
                m_run = m_new;
            }
            const float m_use = (m_run == -INFINITY) ? 0.0f : m_run;
            float p[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                p[i] = fast_exp2(x[i] - m_use);
            const uint32_t pa0 = pack_bf16x2(p[0], p[1]);   // row r, positions cq, cq+1
            const uint32_t pa2 = pack_bf16x2(p[2], p[3]);   // row r, positions 8+cq, 9+cq
            l_run += bf16x2_sum(pa0) + bf16x2_sum(pa2);
#pragma unroll
            for (int dt = 0; dt < D / 16; ++dt) {
                uint32_t v0, v1, v2, v3;
                ldsm_x4_trans(vbase + page_tile_offset<D>(v_row, dt * 16 + v_col, log2p), v0,
                              v1, v2, v3);
                if (n_valid < kKeysPerWarp) {
                    v0 = keep_keys(v0, cq, n_valid);
                    v1 = keep_keys(v1, 8 + cq, n_valid);
                    v2 = keep_keys(v2, cq, n_valid);
                    v3 = keep_keys(v3, 8 + cq, n_valid);
                }
                mma_bf16_16816(o[2 * dt], pa0, 0u, pa2, 0u, v0, v1);
                mma_bf16_16816(o[2 * dt + 1], pa0, 0u, pa2, 0u, v2, v3);
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[st]);
    }
    if (!ok)
        atomicOr(errors, kErrDecodeFullWait);

    // ------------------------- combine the 4 warps' partial results -----------------------
    // Each warp leaves its unnormalised o rows (D + 8 floats apart, so that the rows one store
    // instruction touches fall in distinct banks), running max and row sum; one thread per
    // query head folds them into weights 2^(m_w - M) / L, and the output is written as
    // float4 (bf16x4) pieces.
    constexpr int kRowStride = D + 8;
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    named_barrier(1, kConsumerWarps * 32);   // every warp is done with the ring
    float *red_o = reinterpret_cast<float *>(smem);                      // [W][8][D + 8]
    float *red_m = red_o + kConsumerWarps * kMaxGroup * kRowStride;       // [W][8]
    float *red_l = red_m + kConsumerWarps * kMaxGroup;                    // [W][8]
    float *row_w = red_l + kConsumerWarps * kMaxGroup;                    // [8][W]
    if (r < G) {
        float *dst = red_o + (warp * kMaxGroup + r) * kRowStride + cq;
#pragma unroll
        for (int n = 0; n < D / 8; ++n)
            *reinterpret_cast<float2 *>(dst + n * 8) = make_float2(o[n][0], o[n][1]);
        if ((lane & 3) == 0) {
            red_m[warp * kMaxGroup + r] = m_run;
            red_l[warp * kMaxGroup + r] = l_run;
        }
    }
    named_barrier(1, kConsumerWarps * 32);
    if (threadIdx.x < G) {
        const int row = threadIdx.x;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w)
            M = fmaxf(M, red_m[w * kMaxGroup + row]);
        float f[kConsumerWarps];
        float L = 0.0f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = red_m[w * kMaxGroup + row];
            f[w] = (mw == -INFINITY) ? 0.0f : fast_exp2(mw - M);
            L += f[w] * red_l[w * kMaxGroup + row];
        }
        const float inv = 1.0f / L;   // the chunk holds a valid position: L >= 1
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w)
            row_w[row * kConsumerWarps + w] = f[w] * inv;
        if (SPLIT)
            a.part_lse[(row0 + row) * a.split_stride + a.split_base + split] =
                (M + log2f(L)) * kLn2;
    }
    named_barrier(1, kConsumerWarps * 32);
    constexpr int kVec = D / 4;
    for (int idx = threadIdx.x; idx < G * kVec; idx += kConsumerWarps * 32) {
        const int row = idx / kVec;
        const int c = (idx - row * kVec) * 4;
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float wt = row_w[row * kConsumerWarps + w];
            const float4 v = *reinterpret_cast<const float4 *>(
                red_o + (w * kMaxGroup + row) * kRowStride + c);
            acc.x = fmaf(wt, v.x, acc.x);
            acc.y = fmaf(wt, v.y, acc.y);
            acc.z = fmaf(wt, v.z, acc.z);
            acc.w = fmaf(wt, v.w, acc.w);
        }
        if (SPLIT) {
            const size_t prow = (row0 + row) * a.split_stride + a.split_base + split;
            *reinterpret_cast<float4 *>(a.part_o + prow * D + c) = acc;
        } else {
            store_out4(a.out, a.out_f32, (row0 + row) * D + c, acc);
        }
    }
}

}  // namespace dec
}  // namespace kvc
