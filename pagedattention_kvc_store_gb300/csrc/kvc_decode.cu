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

#include "kvc_decode_cta.cuh"

namespace kvc {

namespace {

__device__ uint32_t g_decode_errors;

using namespace dec;

template <int D, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 2)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const Args a)
{
    pdl_wait();
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    decode_cta<D, SPLIT>(&tmap_k, &tmap_v, a, blockIdx.x, blockIdx.y, blockIdx.z, smem,
                         a.err ? a.err : &g_decode_errors);
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
    const float *po = part_o + static_cast<size_t>(row) * n_split * D + lane * V;
    // The first kPre splits' partials are requested together with the lse values (one memory
    // round trip instead of two on the step's critical path); an empty split's values are
    // loaded but never used.
    constexpr int kPre = 4;
    float pre[kPre][V];
#pragma unroll
    for (int j = 0; j < kPre; ++j) {
        if (j < n_split) {
            if constexpr (V == 4) {
                const float4 t = *reinterpret_cast<const float4 *>(po + static_cast<size_t>(j) * D);
                pre[j][0] = t.x;
                pre[j][1] = t.y;
                pre[j][2] = t.z;
                pre[j][3] = t.w;
            } else {
#pragma unroll
                for (int v = 0; v < V; ++v)
                    pre[j][v] = po[static_cast<size_t>(j) * D + v];
            }
        }
    }
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
        for (int j0 = 0; j0 < n_split; j0 += 32) {
            const float mine = (j0 + lane < n_split) ? lse[j0 + lane] : -INFINITY;
            const int cnt = min(32, n_split - j0);
            for (int jj = 0; jj < cnt; ++jj) {
                const float lj = __shfl_sync(0xffffffffu, mine, jj);
                if (lj == -INFINITY)
                    continue;   // empty split: its partial is not read
                const float w = fast_exp2((lj - M) * kLog2e);
                sum += w;
                const int j = j0 + jj;
                float val[V];
                if (j < kPre) {   // select in registers (no dynamic index into pre)
#pragma unroll
                    for (int k = 0; k < kPre; ++k)
                        if (k == j) {
#pragma unroll
                            for (int v = 0; v < V; ++v)
                                val[v] = pre[k][v];
                        }
                } else if constexpr (V == 4) {
                    const float4 t =
                        *reinterpret_cast<const float4 *>(po + static_cast<size_t>(j) * D);
                    val[0] = t.x;
                    val[1] = t.y;
                    val[2] = t.z;
                    val[3] = t.w;
                } else {
#pragma unroll
                    for (int v = 0; v < V; ++v)
                        val[v] = po[static_cast<size_t>(j) * D + v];
                }
#pragma unroll
                for (int v = 0; v < V; ++v)
                    acc[v] += w * val[v];
            }
        }
    }
    const float inv = (sum > 0.0f) ? 1.0f / sum : 0.0f;
    const size_t base = static_cast<size_t>(row) * D + lane * V;
    if constexpr (V == 4)
        store_out4(out, out_f32, base,
                   make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv));
    else
        store_out2(out, out_f32, base, make_float2(acc[0] * inv, acc[1] * inv));
    if (lse_out != nullptr && lane == 0)
        lse_out[row] = (M == -INFINITY) ? -INFINITY : M + logf(sum);
}

template <int D, bool SPLIT>
cudaError_t launch_decode_t(const DecodeLaunch &l, const CUtensorMap &tk, const CUtensorMap &tv,
                            cudaStream_t stream)
{
    const Args a = make_args(l);
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

// The bounded wait every kernel uses, on an mbarrier phase that nothing completes: it gives
// up after kWaitLimitCycles and the CTA records kErrSelftestWait and returns, leaving the
// context usable.  A diagnostic of the failure path, with no fault and no hang.
__global__ void __launch_bounds__(32) selftest_wait_kernel(uint32_t *word)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (!__all_sync(0xffffffffu, mbar_wait(&bar, 0)) && threadIdx.x == 0)
        atomicOr(word ? word : &g_decode_errors, kErrSelftestWait);
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

cudaError_t launch_selftest_wait(cudaStream_t stream)
{
    selftest_wait_kernel<<<1, 32, 0, stream>>>(current_error_word());
    return cudaGetLastError();
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
