// kvc_decode.cu -- paged decode attention (one new token per sequence, GQA) with a split-K
// partition and the log-sum-exp merge of its partials.
//
// What it computes: "KV Cache Management and PagedAttention", "Compute attention over
// scattered KV" -- attention of the newest token's query over every valid position of its
// sequence, reading K/V in place from the pages its block table lists (no gather buffer),
// excluding unused slots of the last page and every other sequence's pages.  GQA: the G
// query heads of a group share one kv head.
//
// Kernel design (GB300):
//   * one CTA per (split, kv head, sequence); 4 consumer warps + 1 TMA producer warp;
//   * the producer streams 64-position stages of K and V into a 3-deep shared-memory ring
//     with cp.async.bulk.tensor (one box per page, both 64-column halves, 128-byte swizzle so
//     that ldmatrix reads are bank-conflict free), completion counted on mbarriers;
//   * each consumer warp takes 16 of the 64 positions of every stage: S = Q K^T and O += P V
//     on the tensor cores (mma.sync m16n8k16, the G query heads padded to 16 rows -- too thin
//     for tcgen05's 64/128-row tiles), online softmax in base 2 with warp shuffles;
//   * the 4 warps' (max, sum, O) are combined through shared memory at the end; with one
//     split the CTA writes the final output, otherwise an fp32 partial and its lse.
// Masked positions (past the context) are excluded before the exponential and their V
// entries are zeroed in registers, so NaN/Inf left in unused slots never reaches a sum.
#include <math.h>

#include "kvc_device.cuh"
#include "kvc_launch.h"

namespace kvc {

namespace {

__device__ uint32_t g_decode_errors;

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
    static constexpr int kCombineBytes =
        kConsumerWarps * kMaxGroup * (D + 2) * 4;   // o rows + m + l per warp
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
};

__device__ __forceinline__ void store_out(void *out, int out_f32, size_t idx, float v)
{
    if (out_f32)
        static_cast<float *>(out)[idx] = v;
    else
        static_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
}

template <int D, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 2)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const Args a)
{
    pdl_wait();
    pdl_trigger();
    using Geom = DecodeGeom<D>;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Geom::kRingBytes);
    uint64_t *empty = full + kStages;

    const int split = blockIdx.x;
    const int kvh = blockIdx.y;
    const int s = blockIdx.z;
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
    int ctx = a.context_lens[s];
    if (ctx > a.bt_stride * a.page_size) {   // the block-table row cannot hold it
        if (threadIdx.x == 0 && split == 0)
            atomicOr(&g_decode_errors, kErrContextRange);
        ctx = a.bt_stride * a.page_size;
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
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
        }
        const uint64_t policy = l2_policy_evict_first();
        int cached_base = 0;
        int cached_page = pre_page;
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
            const int rel0 = b * kStageKeys;
            const int keys = min(kStageKeys, k_end - k_begin - rel0);
            const int np = (keys + P - 1) / P;
            if (lane == 0)
                mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(np * P * D * 2 * 2));
            __syncwarp();
            uint8_t *kdst = smem + st * Geom::kStageBytes;
            uint8_t *vdst = kdst + Geom::kTileBytes;
            const int lp0 = rel0 / P;   // first page of the stage inside this chunk
            if (lp0 + np > cached_base + 32) {
                cached_base = lp0;
                cached_page = (lp0 + lane < n_pages) ? bt_row[lp0 + lane] : 0;
            }
            // Lane 2 i loads page i of K, lane 2 i + 1 page i of V: boxes issued together by
            // several lanes reach a much higher TMA rate than one thread issuing them in turn.
            const int i = lane >> 1;
            const int page = __shfl_sync(0xffffffffu, cached_page, (lp0 - cached_base + i) & 31);
            if (i < np) {
                const int off = i * P * D * 2;
                // NHD maps {64, slot, half, kv head}; HND maps {64, offset, half, block}
                const int c1 = a.hnd ? 0 : page * P;
                const int c3 = a.hnd ? page * a.kv_heads + kvh : kvh;
                if (lane & 1)
                    tma_load_4d_hint(vdst + off, &tmap_v, 0, c1, 0, c3, &full[st], policy);
                else
                    tma_load_4d_hint(kdst + off, &tmap_k, 0, c1, 0, c3, &full[st], policy);
            }
            issued = b + 1;
        }
        if (!ok && lane == 0) {
            atomicOr(&g_decode_errors, kErrDecodeEmptyWait);
            // Let every copy already in flight land before the CTA can exit.
            for (int b = max(0, issued - kStages); b < issued; ++b)
                if (!mbar_wait(&full[b % kStages], (b / kStages) & 1))
                    atomicOr(&g_decode_errors, kErrDrainWait);
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
        atomicOr(&g_decode_errors, kErrDecodeFullWait);

    // ------------------------- combine the 4 warps' partial results -----------------------
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    named_barrier(1, kConsumerWarps * 32);   // every warp is done with the ring
    float *red_o = reinterpret_cast<float *>(smem);                      // [W][8][D]
    float *red_m = red_o + kConsumerWarps * kMaxGroup * D;                // [W][8]
    float *red_l = red_m + kConsumerWarps * kMaxGroup;                    // [W][8]
    if (r < G) {
        float *dst = red_o + (warp * kMaxGroup + r) * D;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            dst[n * 8 + cq] = o[n][0];
            dst[n * 8 + cq + 1] = o[n][1];
        }
        if ((lane & 3) == 0) {
            red_m[warp * kMaxGroup + r] = m_run;
            red_l[warp * kMaxGroup + r] = l_run;
        }
    }
    named_barrier(1, kConsumerWarps * 32);
    for (int idx = threadIdx.x; idx < G * D; idx += kConsumerWarps * 32) {
        const int row = idx / D;
        const int d = idx - row * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w)
            M = fmaxf(M, red_m[w * kMaxGroup + row]);
        float L = 0.0f, O = 0.0f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = red_m[w * kMaxGroup + row];
            const float f = (mw == -INFINITY) ? 0.0f : fast_exp2(mw - M);
            L += f * red_l[w * kMaxGroup + row];
            O += f * red_o[(w * kMaxGroup + row) * D + d];
        }
        const float val = O / L;
        if (SPLIT) {
            const size_t prow = (row0 + row) * a.split_stride + a.split_base + split;
            a.part_o[prow * D + d] = val;
            if (d == 0)
                a.part_lse[prow] = (M + log2f(L)) * kLn2;
        } else {
            store_out(a.out, a.out_f32, (row0 + row) * D + d, val);
        }
    }
}

// One warp per row: out[r] = sum_j exp(lse_j - M) o_j / sum_j exp(lse_j - M).
template <int D>
__global__ void __launch_bounds__(128) merge_kernel(void *out, int out_f32,
                                                    const float *__restrict__ part_o,
                                                    const float *__restrict__ part_lse,
                                                    int rows, int n_split, float *lse_out)
{
    pdl_wait();
    pdl_trigger();
    constexpr int V = D / 32;
    const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows)
        return;
    const float *lse = part_lse + static_cast<size_t>(row) * n_split;
    float M = -INFINITY;
    for (int j = lane; j < n_split; j += 32)
        M = fmaxf(M, lse[j]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v)
        acc[v] = 0.0f;
    float sum = 0.0f;
    if (M != -INFINITY) {
        const float *po = part_o + static_cast<size_t>(row) * n_split * D + lane * V;
        for (int j0 = 0; j0 < n_split; j0 += 32) {
            const float mine = (j0 + lane < n_split) ? lse[j0 + lane] : -INFINITY;
            const int cnt = min(32, n_split - j0);
            for (int jj = 0; jj < cnt; ++jj) {
                const float lj = __shfl_sync(0xffffffffu, mine, jj);
                if (lj == -INFINITY)
                    continue;   // empty split: its partial is not read
                const float w = fast_exp2((lj - M) * kLog2e);
                sum += w;
                const float *src = po + static_cast<size_t>(j0 + jj) * D;
                if constexpr (V == 4) {
                    const float4 val = *reinterpret_cast<const float4 *>(src);
                    acc[0] += w * val.x;
                    acc[1] += w * val.y;
                    acc[2] += w * val.z;
                    acc[3] += w * val.w;
                } else {
#pragma unroll
                    for (int v = 0; v < V; ++v)
                        acc[v] += w * src[v];
                }
            }
        }
    }
    const float inv = (sum > 0.0f) ? 1.0f / sum : 0.0f;
    const size_t base = static_cast<size_t>(row) * D + lane * V;
#pragma unroll
    for (int v = 0; v < V; ++v)
        store_out(out, out_f32, base + v, acc[v] * inv);
    if (lse_out != nullptr && lane == 0)
        lse_out[row] = (M == -INFINITY) ? -INFINITY : M + logf(sum);
}

template <int D, bool SPLIT>
cudaError_t launch_decode_t(const DecodeLaunch &l, const CUtensorMap &tk, const CUtensorMap &tv,
                            cudaStream_t stream)
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
    const size_t smem = DecodeGeom<D>::kSmemBytes;
    auto kernel = paged_decode_kernel<D, SPLIT>;
    cudaError_t err =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (err != cudaSuccess)
        return err;
    dim3 grid(l.n_split, l.kv_heads, l.num_seqs);
    return launch_pdl(kernel, grid, dim3(kThreads), smem, stream, tk, tv, a);
}

}  // namespace

cudaError_t launch_decode(const DecodeLaunch &l, const CUtensorMap &tk, const CUtensorMap &tv,
                          cudaStream_t stream)
{
    if (l.num_seqs == 0)
        return cudaSuccess;
    const bool split = l.n_split > 1 || l.split_stride > 1 || l.key_start != nullptr;
    if (l.head_dim == 128)
        return split ? launch_decode_t<128, true>(l, tk, tv, stream)
                     : launch_decode_t<128, false>(l, tk, tv, stream);
    return split ? launch_decode_t<64, true>(l, tk, tv, stream)
                 : launch_decode_t<64, false>(l, tk, tv, stream);
}

cudaError_t launch_merge(void *out, int out_f32, const float *part_o, const float *part_lse,
                         int rows, int n_split, int head_dim, float *lse_out,
                         cudaStream_t stream)
{
    if (rows == 0)
        return cudaSuccess;
    const int blocks = (rows + 3) / 4;
    if (head_dim == 128)
        return launch_pdl(merge_kernel<128>, dim3(blocks), dim3(128), 0, stream, out, out_f32,
                          part_o, part_lse, rows, n_split, lse_out);
    return launch_pdl(merge_kernel<64>, dim3(blocks), dim3(128), 0, stream, out, out_f32, part_o,
                      part_lse, rows, n_split, lse_out);
}

cudaError_t read_and_clear_decode_errors(uint32_t *flags)
{
    uint32_t zero = 0;
    cudaError_t err = cudaMemcpyFromSymbol(flags, g_decode_errors, sizeof(uint32_t));
    if (err != cudaSuccess)
        return err;
    return cudaMemcpyToSymbol(g_decode_errors, &zero, sizeof(uint32_t));
}

}  // namespace kvc
