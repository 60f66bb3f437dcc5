// kvc_append.cu -- causal chunked prefill over a paged, already-cached prefix.
//
// What it computes: Quail "KV", "KV rewind" (a question appended after a cached document)
// and "Prefix sharing"; TileInfer.jl "KV cache", "Prefix reuse in chat".  New token i of a
// sequence with ctx positions and q_len new tokens sits at position ctx - q_len + i and
// attends, causally, to positions 0 .. ctx - q_len + i -- the cached prefix plus the new
// tokens before it and itself -- read in place from the pages of its block table.
//
// Kernel design (mma.sync path):
//   * rows of the attention problem are (new token, query head of the GQA group) pairs,
//     token-major, so one kv head's K/V tile feeds G * tokens rows at once;
//   * one CTA per (64-row block, kv head, sequence): 4 consumer warps of 16 rows each and
//     one TMA producer warp streaming 64-position K/V stages through a 3-deep ring (same
//     swizzled layout as decode); the producer walks the block table 32 entries at a time;
//   * S = Q K^T and O += P V on mma.sync m16n8k16 (bf16 in, fp32 accumulate), online
//     softmax in base 2; the causal limit of each row is applied before the exponential.
#include <math.h>

#include "kvc_device.cuh"
#include "kvc_launch.h"

namespace kvc {

namespace {

__device__ uint32_t g_append_errors;

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 3;
constexpr int kRowsPerWarp = 16;
constexpr int kRowsPerCta = kConsumerWarps * kRowsPerWarp;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct AppendGeom {
    static constexpr int kTileBytes = (D / 64) * kStageKeys * 128;
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr size_t kSmemBytes = 1024 + kRingBytes + 2 * kStages * 8;
};

struct Args {
    const __nv_bfloat16 *q;
    void *out;
    int out_f32;
    const int32_t *block_table;
    int bt_stride;
    const int32_t *q_indptr;
    const int32_t *context_lens;
    int q_heads, group, page_size;
    float scale_log2;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    paged_append_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const Args a)
{
    using Geom = AppendGeom<D>;
    constexpr int kHalves = D / 64;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Geom::kRingBytes);
    uint64_t *empty = full + kStages;

    const int mb = blockIdx.x;
    const int kvh = blockIdx.y;
    const int s = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.group;
    const int P = a.page_size;
    const int tok0 = a.q_indptr[s];
    const int q_len = a.q_indptr[s + 1] - tok0;
    int ctx = a.context_lens[s];
    if (ctx > a.bt_stride * P) {   // the block-table row cannot hold it
        if (threadIdx.x == 0 && mb == 0)
            atomicOr(&g_append_errors, kErrContextRange);
        ctx = a.bt_stride * P;
    }
    const int rows = q_len * G;
    const int row_begin = mb * kRowsPerCta;
    if (row_begin >= rows)
        return;
    const int row_last = min(rows, row_begin + kRowsPerCta) - 1;
    // keys this CTA needs: 0 .. (position of its last token)
    const int n_keys = min(ctx, ctx - q_len + row_last / G + 1);
    if (n_keys <= 0)
        return;   // malformed (ctx < q_len); nothing visible
    const int n_blocks = (n_keys + kStageKeys - 1) / kStageKeys;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // --------------------------- TMA producer (whole warp) ----------------------------
        const int32_t *bt_row = a.block_table + static_cast<size_t>(s) * a.bt_stride;
        const int n_pages = (n_keys + P - 1) / P;
        if (lane == 0) {
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
        }
        const uint64_t policy = l2_policy_evict_last();   // K/V are re-read by sibling CTAs
        int cached_base = -32;
        int cached_page = 0;
        int issued = 0;
        bool ok = true;
        for (int b = 0; b < n_blocks; ++b) {
            const int st = b % kStages;
            if (b >= kStages) {
                const bool waited = mbar_wait(&empty[st], ((b / kStages) - 1) & 1);
                if (!__all_sync(0xffffffffu, waited)) {
                    ok = false;
                    break;
                }
            }
            const int key0 = b * kStageKeys;
            const int np = (min(kStageKeys, n_keys - key0) + P - 1) / P;
            if (lane == 0)
                mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(np * P * D * 2 * 2));
            uint8_t *kdst = smem + st * Geom::kStageBytes;
            uint8_t *vdst = kdst + Geom::kTileBytes;
            for (int i = 0; i < np; ++i) {
                const int lp = key0 / P + i;   // logical page
                if (lp >= cached_base + 32) {
                    cached_base = lp;
                    cached_page = (lp + lane < n_pages) ? bt_row[lp + lane] : 0;
                }
                const int page = __shfl_sync(0xffffffffu, cached_page, lp - cached_base);
                if (lane == 0) {
                    const int slot0 = page * P;
#pragma unroll
                    for (int h = 0; h < kHalves; ++h) {
                        const int off = h * kStageKeys * 128 + i * P * 128;
                        tma_load_3d(kdst + off, &tmap_k, h * 64, kvh, slot0, &full[st], policy);
                        tma_load_3d(vdst + off, &tmap_v, h * 64, kvh, slot0, &full[st], policy);
                    }
                }
            }
            issued = b + 1;
        }
        if (!ok && lane == 0) {
            atomicOr(&g_append_errors, kErrAppendEmptyWait);
            for (int b = max(0, issued - kStages); b < issued; ++b)
                if (!mbar_wait(&full[b % kStages], (b / kStages) & 1))
                    atomicOr(&g_append_errors, kErrDrainWait);
        }
        return;
    }

    // ----------------------------------- consumers ----------------------------------------
    const int cq = (lane & 3) * 2;
    const int ra = row_begin + warp * kRowsPerWarp + (lane >> 2);   // fragment rows ra, ra + 8
    const int rb = ra + 8;
    const bool va = ra < rows, vb = rb < rows;
    const int ia = ra / G, ga = ra - ia * G;
    const int ib = rb / G, gb = rb - ib * G;
    // last visible key of each row (-1: padding row, sees nothing)
    const int lim_a = va ? ctx - q_len + ia : -1;
    const int lim_b = vb ? ctx - q_len + ib : -1;
    int lim_min = min(lim_a, lim_b);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        lim_min = min(lim_min, __shfl_xor_sync(0xffffffffu, lim_min, off));

    const size_t qrow_a = (static_cast<size_t>(tok0 + ia) * a.q_heads + kvh * G + ga) * D;
    const size_t qrow_b = (static_cast<size_t>(tok0 + ib) * a.q_heads + kvh * G + gb) * D;
    uint32_t qa[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const int c = kk * 16 + cq;
        qa[kk][0] = va ? *reinterpret_cast<const uint32_t *>(a.q + qrow_a + c) : 0u;
        qa[kk][1] = vb ? *reinterpret_cast<const uint32_t *>(a.q + qrow_b + c) : 0u;
        qa[kk][2] = va ? *reinterpret_cast<const uint32_t *>(a.q + qrow_a + c + 8) : 0u;
        qa[kk][3] = vb ? *reinterpret_cast<const uint32_t *>(a.q + qrow_b + c + 8) : 0u;
    }
    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
        o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.0f, l_b = 0.0f;

    const int k_row = (lane & 7) + ((lane >> 4) << 3);
    const int k_col = ((lane >> 3) & 1) << 3;
    const int v_row = (lane & 7) + (((lane >> 3) & 1) << 3);
    const int v_col = (lane >> 4) << 3;
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
        const int key0 = b * kStageKeys;
        const int n_valid = n_keys - key0;   // positions of this stage holding loaded data

        float sc[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n)
            sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.0f;
#pragma unroll
        for (int pr = 0; pr < 4; ++pr) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kbase + swz_offset<kStageKeys>(pr * 16 + k_row, kk * 16 + k_col), b0, b1,
                        b2, b3);
                mma_bf16_16816(sc[2 * pr], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                mma_bf16_16816(sc[2 * pr + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2,
                               b3);
            }
        }
        // scale, causal mask, row max
        const bool need_mask = key0 + kStageKeys - 1 > lim_min;
        float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float xa = sc[n][e] * sl2;
                float xb = sc[n][2 + e] * sl2;
                if (need_mask) {
                    const int key = key0 + n * 8 + cq + e;
                    if (key > lim_a)
                        xa = -INFINITY;
                    if (key > lim_b)
                        xb = -INFINITY;
                }
                sc[n][e] = xa;
                sc[n][2 + e] = xb;
                mx_a = fmaxf(mx_a, xa);
                mx_b = fmaxf(mx_b, xb);
            }
        }
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
        const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
        if (__any_sync(0xffffffffu, (mn_a > m_a) || (mn_b > m_b))) {
            const float al_a = (m_a == -INFINITY) ? 0.0f : fast_exp2(m_a - mn_a);
            const float al_b = (m_b == -INFINITY) ? 0.0f : fast_exp2(m_b - mn_b);
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
                o[n][0] *= al_a;
                o[n][1] *= al_a;
                o[n][2] *= al_b;
                o[n][3] *= al_b;
            }
            l_a *= al_a;
            l_b *= al_b;
            m_a = mn_a;
            m_b = mn_b;
        }
        const float mu_a = (m_a == -INFINITY) ? 0.0f : m_a;
        const float mu_b = (m_b == -INFINITY) ? 0.0f : m_b;
        uint32_t pa[8][2];
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            pa[n][0] = pack_bf16x2(fast_exp2(sc[n][0] - mu_a), fast_exp2(sc[n][1] - mu_a));
            pa[n][1] = pack_bf16x2(fast_exp2(sc[n][2] - mu_b), fast_exp2(sc[n][3] - mu_b));
            l_a += bf16x2_sum(pa[n][0]);
            l_b += bf16x2_sum(pa[n][1]);
        }
        // O += P V, 16 positions per k-step
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            if (ks * 16 >= n_valid)
                break;
#pragma unroll
            for (int dt = 0; dt < D / 16; ++dt) {
                uint32_t v0, v1, v2, v3;
                ldsm_x4_trans(vbase + swz_offset<kStageKeys>(ks * 16 + v_row, dt * 16 + v_col),
                              v0, v1, v2, v3);
                if (n_valid < (ks + 1) * 16) {
                    v0 = keep_keys(v0, ks * 16 + cq, n_valid);
                    v1 = keep_keys(v1, ks * 16 + 8 + cq, n_valid);
                    v2 = keep_keys(v2, ks * 16 + cq, n_valid);
                    v3 = keep_keys(v3, ks * 16 + 8 + cq, n_valid);
                }
                mma_bf16_16816(o[2 * dt], pa[2 * ks][0], pa[2 * ks][1], pa[2 * ks + 1][0],
                               pa[2 * ks + 1][1], v0, v1);
                mma_bf16_16816(o[2 * dt + 1], pa[2 * ks][0], pa[2 * ks][1], pa[2 * ks + 1][0],
                               pa[2 * ks + 1][1], v2, v3);
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[st]);
    }
    if (!ok)
        atomicOr(&g_append_errors, kErrAppendFullWait);

    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    const float inv_a = l_a > 0.0f ? 1.0f / l_a : 0.0f;
    const float inv_b = l_b > 0.0f ? 1.0f / l_b : 0.0f;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
        const int d = n * 8 + cq;
        if (va) {
            const size_t idx = qrow_a + d;
            if (a.out_f32) {
                *reinterpret_cast<float2 *>(static_cast<float *>(a.out) + idx) =
                    make_float2(o[n][0] * inv_a, o[n][1] * inv_a);
            } else {
                *reinterpret_cast<uint32_t *>(static_cast<__nv_bfloat16 *>(a.out) + idx) =
                    pack_bf16x2(o[n][0] * inv_a, o[n][1] * inv_a);
            }
        }
        if (vb) {
            const size_t idx = qrow_b + d;
            if (a.out_f32) {
                *reinterpret_cast<float2 *>(static_cast<float *>(a.out) + idx) =
                    make_float2(o[n][2] * inv_b, o[n][3] * inv_b);
            } else {
                *reinterpret_cast<uint32_t *>(static_cast<__nv_bfloat16 *>(a.out) + idx) =
                    pack_bf16x2(o[n][2] * inv_b, o[n][3] * inv_b);
            }
        }
    }
}

template <int D>
cudaError_t launch_append_t(const AppendLaunch &l, const CUtensorMap &tk, const CUtensorMap &tv,
                            cudaStream_t stream)
{
    Args a;
    a.q = static_cast<const __nv_bfloat16 *>(l.q);
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
    const size_t smem = AppendGeom<D>::kSmemBytes;
    auto kernel = paged_append_kernel<D>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess)
        return err;
    const int m_blocks = (l.max_q_len * a.group + kRowsPerCta - 1) / kRowsPerCta;
    dim3 grid(m_blocks, l.kv_heads, l.num_seqs);
    kernel<<<grid, kThreads, smem, stream>>>(tk, tv, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append(const AppendLaunch &l, const CUtensorMap &tk, const CUtensorMap &tv,
                          cudaStream_t stream)
{
    if (l.num_seqs == 0 || l.num_tokens == 0 || l.max_q_len == 0)
        return cudaSuccess;
    return l.head_dim == 128 ? launch_append_t<128>(l, tk, tv, stream)
                             : launch_append_t<64>(l, tk, tv, stream);
}

cudaError_t read_and_clear_append_errors(uint32_t *flags)
{
    uint32_t zero = 0;
    cudaError_t err = cudaMemcpyFromSymbol(flags, g_append_errors, sizeof(uint32_t));
    if (err != cudaSuccess)
        return err;
    return cudaMemcpyToSymbol(g_append_errors, &zero, sizeof(uint32_t));
}

}  // namespace kvc
