// kvc_grouped.cu -- decode for groups of sequences that share a prefix of pages.
//
// What it computes: the same attention as kvc_decode ("KV Cache Management and
// PagedAttention", "Compute attention over scattered KV"), for sequences whose block tables
// begin with the same physical pages ("Share common KV across responses"; Quail "KV",
// "Prefix sharing").  Each response still attends with its own query over its own context;
// only the reading of the shared pages is done once per group instead of once per member.
//
// Decomposition (all partials are normalised fp32 pieces with their log-sum-exp):
//   prefix  one CTA per (prefix chunk, kv head, group): the chunk's pages, read once, against
//           the query rows of every member of the group (members x G rows, at most 64), on
//           mma.sync tiles of 16 rows -- this kernel;
//   suffix  each member's positions from the end of the prefix, with the decode kernel
//           (kvc_decode.cu, started at key_start[s]);
//   merge   log-sum-exp over prefix and suffix partials (merge_kernel).
// A TMA producer warp streams the prefix pages (one box per page) into a 3-deep swizzled
// ring; four consumer warps cover 1, 2 or 4 row tiles, the warps of one tile splitting each
// 64-position stage between them and combining through shared memory at the end.
#include <math.h>

#include "kvc_device.cuh"
#include "kvc_launch.h"

namespace kvc {

namespace {

__device__ uint32_t g_grouped_errors;

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 3;
constexpr int kMaxRows = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct GroupGeom {
    static constexpr int kTileBytes = kStageKeys * D * 2;
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kCombineBytes = kConsumerWarps * 16 * (D + 2) * 4;
    static_assert(kCombineBytes <= kRingBytes, "combine area aliases the ring");
    static constexpr size_t kSmemBytes = 1024 + kRingBytes + 2 * kStages * 8;
};

struct Args {
    const __nv_bfloat16 *q;
    float *part_o;
    float *part_lse;
    const int32_t *block_table;
    int bt_stride;
    const int32_t *group_indptr;
    const int32_t *group_seqs;
    const int32_t *prefix_len;
    int q_heads, kv_heads, group, page_size;
    int chunk, split_stride;
    float scale_log2;
    int hnd;   // HND pools: page boxes addressed by (page, kv head) block
};

__global__ void grouped_setup_kernel(float *__restrict__ part_lse, int32_t *__restrict__ key_start,
                                     int num_seqs, int q_heads, int n_prefix, int split_stride)
{
    pdl_wait();
    pdl_trigger();
    const size_t total = static_cast<size_t>(num_seqs) * q_heads * n_prefix;
    const size_t step = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += step) {
        const size_t row = i / n_prefix;
        const size_t j = i - row * n_prefix;
        part_lse[row * split_stride + j] = -INFINITY;
    }
    for (size_t s = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
         s < static_cast<size_t>(num_seqs); s += step)
        key_start[s] = 0;
}

__global__ void grouped_members_kernel(int32_t *__restrict__ key_start,
                                       const int32_t *__restrict__ group_indptr,
                                       const int32_t *__restrict__ group_seqs,
                                       const int32_t *__restrict__ prefix_len, int page_size,
                                       int bt_stride)
{
    pdl_wait();
    pdl_trigger();
    const int g = blockIdx.x;
    int pre = (prefix_len[g] / page_size) * page_size;   // whole pages only
    pre = min(max(pre, 0), bt_stride * page_size);
    for (int i = group_indptr[g] + threadIdx.x; i < group_indptr[g + 1]; i += blockDim.x)
        key_start[group_seqs[i]] = pre;
}

template <int D, int NMT>
__global__ void __launch_bounds__(kThreads, 2)
    grouped_prefix_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, const Args a)
{
    pdl_wait();
    pdl_trigger();
    using Geom = GroupGeom<D>;
    constexpr int kWarpsPerTile = kConsumerWarps / NMT;   // warps sharing one 16-row tile
    constexpr int kKeysPerWarp = kStageKeys / kWarpsPerTile;
    constexpr int kNT = kKeysPerWarp / 8;                  // n-tiles of S per warp and stage

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Geom::kRingBytes);
    uint64_t *empty = full + kStages;

    const int split = blockIdx.x;
    const int kvh = blockIdx.y;
    const int grp = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.group;
    const int P = a.page_size;
    const int m0 = a.group_indptr[grp];
    const int rows = min((a.group_indptr[grp + 1] - m0) * G, NMT * 16);
    int prefix = (a.prefix_len[grp] / P) * P;
    prefix = min(max(prefix, 0), a.bt_stride * P);
    const int k_begin = split * a.chunk;
    const int k_end = min(prefix, k_begin + a.chunk);
    if (k_begin >= k_end || rows <= 0)
        return;   // the setup kernel already marked this split empty for every row
    const int leader = a.group_seqs[m0];
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
        const int32_t *bt_row =
            a.block_table + static_cast<size_t>(leader) * a.bt_stride + first_page;
        if (lane == 0) {
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
        }
        const uint64_t policy = l2_policy_evict_first();
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
            atomicOr(&g_grouped_errors, kErrDecodeEmptyWait);
            for (int b = max(0, issued - kStages); b < issued; ++b)
                if (!mbar_wait(&full[b % kStages], (b / kStages) & 1))
                    atomicOr(&g_grouped_errors, kErrDrainWait);
        }
        return;
    }

    // --------------------------------- consumers -----------------------------------------
    const int mt = warp / kWarpsPerTile;   // this warp's 16-row tile
    const int ksl = warp % kWarpsPerTile;  // its slice of every stage's positions
    const int cq = (lane & 3) * 2;
    const int ra = mt * 16 + (lane >> 2);  // fragment rows ra and ra + 8
    const int rb = ra + 8;
    const bool va = ra < rows, vb = rb < rows;
    auto q_row_ptr = [&](int r) {
        const int m = r / G;
        const int gh = r - m * G;
        const int seq = a.group_seqs[m0 + m];
        return a.q + (static_cast<size_t>(seq) * a.q_heads + static_cast<size_t>(kvh) * G + gh) * D;
    };
    uint32_t qa[D / 16][4];
    {
        const __nv_bfloat16 *qa_row = va ? q_row_ptr(ra) : nullptr;
        const __nv_bfloat16 *qb_row = vb ? q_row_ptr(rb) : nullptr;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int c = kk * 16 + cq;
            qa[kk][0] = va ? *reinterpret_cast<const uint32_t *>(qa_row + c) : 0u;
            qa[kk][1] = vb ? *reinterpret_cast<const uint32_t *>(qb_row + c) : 0u;
            qa[kk][2] = va ? *reinterpret_cast<const uint32_t *>(qa_row + c + 8) : 0u;
            qa[kk][3] = vb ? *reinterpret_cast<const uint32_t *>(qb_row + c + 8) : 0u;
        }
    }
    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
        o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.0f, l_b = 0.0f;

    const int log2p = __ffs(P) - 1;
    const int k_row = ksl * kKeysPerWarp + (lane & 7) + ((lane >> 4) << 3);
    const int k_col = ((lane >> 3) & 1) << 3;
    const int v_row = ksl * kKeysPerWarp + (lane & 7) + (((lane >> 3) & 1) << 3);
    const int v_col = (lane >> 4) << 3;
    const float sl2 = a.scale_log2;
    bool ok = true;

    for (int b = 0; b < n_blocks; ++b) {
        const int st = b % kStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&full[st], (b / kStages) & 1))) {
            ok = false;
            break;
        }
        const uint32_t kbase = smem_addr(smem + st * Geom::kStageBytes);
        const uint32_t vbase = kbase + Geom::kTileBytes;
        const int n_valid = k_end - (k_begin + b * kStageKeys + ksl * kKeysPerWarp);
        if (n_valid > 0) {
            float sc[kNT][4];
#pragma unroll
            for (int n = 0; n < kNT; ++n)
                sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.0f;
#pragma unroll
            for (int pr = 0; pr < kNT / 2; ++pr) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kbase + page_tile_offset<D>(pr * 16 + k_row, kk * 16 + k_col, log2p),
                            b0, b1, b2, b3);
                    mma_bf16_16816(sc[2 * pr], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0,
                                   b1);
                    mma_bf16_16816(sc[2 * pr + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3],
                                   b2, b3);
                }
            }
            float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
            for (int n = 0; n < kNT; ++n) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    if (n * 8 + cq + e >= n_valid) {
                        sc[n][e] = -INFINITY;
                        sc[n][2 + e] = -INFINITY;
                    }
                    mx_a = fmaxf(mx_a, sc[n][e]);
                    mx_b = fmaxf(mx_b, sc[n][2 + e]);
                }
            }
            mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
            mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
            mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
            mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
            const float mn_a = fmaxf(m_a, mx_a * sl2), mn_b = fmaxf(m_b, mx_b * sl2);
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
            const float nu_a = (m_a == -INFINITY) ? 0.0f : -m_a;
            const float nu_b = (m_b == -INFINITY) ? 0.0f : -m_b;
            uint32_t pa[kNT][2];
#pragma unroll
            for (int n = 0; n < kNT; ++n) {
                pa[n][0] = pack_bf16x2(fast_exp2(fmaf(sc[n][0], sl2, nu_a)),
                                       fast_exp2(fmaf(sc[n][1], sl2, nu_a)));
                pa[n][1] = pack_bf16x2(fast_exp2(fmaf(sc[n][2], sl2, nu_b)),
                                       fast_exp2(fmaf(sc[n][3], sl2, nu_b)));
                l_a += bf16x2_sum(pa[n][0]);
                l_b += bf16x2_sum(pa[n][1]);
            }
#pragma unroll
            for (int ks = 0; ks < kKeysPerWarp / 16; ++ks) {
                if (ks * 16 >= n_valid)
                    break;
#pragma unroll
                for (int dt = 0; dt < D / 16; ++dt) {
                    uint32_t v0, v1, v2, v3;
                    ldsm_x4_trans(vbase + page_tile_offset<D>(ks * 16 + v_row, dt * 16 + v_col,
                                                              log2p),
                                  v0, v1, v2, v3);
                    if (n_valid < (ks + 1) * 16) {
                        v0 = keep_keys(v0, ks * 16 + cq, n_valid);
                        v1 = keep_keys(v1, ks * 16 + 8 + cq, n_valid);
                        v2 = keep_keys(v2, ks * 16 + cq, n_valid);
                        v3 = keep_keys(v3, ks * 16 + 8 + cq, n_valid);
                    }
                    mma_bf16_16816(o[2 * dt], pa[2 * ks][0], pa[2 * ks][1], pa[2 * ks + 1][0],
                                   pa[2 * ks + 1][1], v0, v1);
                    mma_bf16_16816(o[2 * dt + 1], pa[2 * ks][0], pa[2 * ks][1],
                                   pa[2 * ks + 1][0], pa[2 * ks + 1][1], v2, v3);
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[st]);
    }
    if (!ok)
        atomicOr(&g_grouped_errors, kErrDecodeFullWait);

    // ------------------- combine the warps of each tile, write partials --------------------
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    named_barrier(1, kConsumerWarps * 32);   // every warp is done with the ring
    float *red_o = reinterpret_cast<float *>(smem);                    // [W][16][D]
    float *red_m = red_o + kConsumerWarps * 16 * D;                     // [W][16]
    float *red_l = red_m + kConsumerWarps * 16;                         // [W][16]
    {
        const int la = lane >> 2, lb = la + 8;
        float *dst_a = red_o + (warp * 16 + la) * D;
        float *dst_b = red_o + (warp * 16 + lb) * D;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            dst_a[n * 8 + cq] = o[n][0];
            dst_a[n * 8 + cq + 1] = o[n][1];
            dst_b[n * 8 + cq] = o[n][2];
            dst_b[n * 8 + cq + 1] = o[n][3];
        }
        if ((lane & 3) == 0) {
            red_m[warp * 16 + la] = m_a;
            red_l[warp * 16 + la] = l_a;
            red_m[warp * 16 + lb] = m_b;
            red_l[warp * 16 + lb] = l_b;
        }
    }
    named_barrier(1, kConsumerWarps * 32);
    for (int idx = threadIdx.x; idx < rows * D; idx += kConsumerWarps * 32) {
        const int r = idx / D;
        const int d = idx - r * D;
        const int tile = r >> 4;
        const int rr = r & 15;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarpsPerTile; ++w)
            M = fmaxf(M, red_m[(tile * kWarpsPerTile + w) * 16 + rr]);
        float L = 0.0f, O = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarpsPerTile; ++w) {
            const int slot = (tile * kWarpsPerTile + w) * 16 + rr;
            const float mw = red_m[slot];
            const float f = (mw == -INFINITY) ? 0.0f : fast_exp2(mw - M);
            L += f * red_l[slot];
            O += f * red_o[slot * D + d];
        }
        const int m = r / G;
        const int gh = r - m * G;
        const int seq = a.group_seqs[m0 + m];
        const size_t prow =
            (static_cast<size_t>(seq) * a.q_heads + static_cast<size_t>(kvh) * G + gh) *
                a.split_stride + split;
        a.part_o[prow * D + d] = (L > 0.0f) ? O / L : 0.0f;
        if (d == 0)
            a.part_lse[prow] = (L > 0.0f) ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
}

template <int D, int NMT>
cudaError_t launch_t(const GroupedPrefixLaunch &l, const CUtensorMap &tk, const CUtensorMap &tv,
                     cudaStream_t stream)
{
    Args a;
    a.q = static_cast<const __nv_bfloat16 *>(l.q);
    a.part_o = l.part_o;
    a.part_lse = l.part_lse;
    a.block_table = l.block_table;
    a.bt_stride = l.bt_stride;
    a.group_indptr = l.group_indptr;
    a.group_seqs = l.group_seqs;
    a.prefix_len = l.prefix_len;
    a.q_heads = l.q_heads;
    a.kv_heads = l.kv_heads;
    a.hnd = l.hnd ? 1 : 0;
    a.group = l.q_heads / l.kv_heads;
    a.page_size = l.page_size;
    a.chunk = l.chunk;
    a.split_stride = l.split_stride;
    a.scale_log2 = l.scale * kLog2e;
    const size_t smem = GroupGeom<D>::kSmemBytes;
    auto kernel = grouped_prefix_kernel<D, NMT>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess)
        return err;
    dim3 grid(l.n_split, l.kv_heads, l.num_groups);
    return launch_pdl(kernel, grid, dim3(kThreads), smem, stream, tk, tv, a);
}

template <int D>
cudaError_t launch_d(const GroupedPrefixLaunch &l, const CUtensorMap &tk, const CUtensorMap &tv,
                     cudaStream_t stream)
{
    if (l.max_rows <= 16)
        return launch_t<D, 1>(l, tk, tv, stream);
    if (l.max_rows <= 32)
        return launch_t<D, 2>(l, tk, tv, stream);
    return launch_t<D, 4>(l, tk, tv, stream);
}

}  // namespace

cudaError_t launch_grouped_setup(float *part_lse, int32_t *key_start, const int32_t *group_indptr,
                                 const int32_t *group_seqs, const int32_t *prefix_len,
                                 int num_groups, int num_seqs, int q_heads, int n_prefix_splits,
                                 int split_stride, int page_size, int bt_stride,
                                 cudaStream_t stream)
{
    const size_t total = static_cast<size_t>(num_seqs) * q_heads * n_prefix_splits;
    const size_t want = (total + 255) / 256;
    const int blocks = static_cast<int>(want < 1024 ? (want > 0 ? want : 1) : 1024);
    cudaError_t err = launch_pdl(grouped_setup_kernel, dim3(blocks), dim3(256), 0, stream,
                                 part_lse, key_start, num_seqs, q_heads, n_prefix_splits,
                                 split_stride);
    if (err == cudaSuccess && num_groups > 0)
        err = launch_pdl(grouped_members_kernel, dim3(num_groups), dim3(128), 0, stream,
                         key_start, group_indptr, group_seqs, prefix_len, page_size, bt_stride);
    return err;
}

cudaError_t launch_grouped_prefix(const GroupedPrefixLaunch &l, const CUtensorMap &tk,
                                  const CUtensorMap &tv, cudaStream_t stream)
{
    if (l.num_groups == 0 || l.n_split == 0)
        return cudaSuccess;
    return l.head_dim == 128 ? launch_d<128>(l, tk, tv, stream) : launch_d<64>(l, tk, tv, stream);
}

cudaError_t read_and_clear_grouped_errors(uint32_t *flags)
{
    uint32_t zero = 0;
    cudaError_t err = cudaMemcpyFromSymbol(flags, g_grouped_errors, sizeof(uint32_t));
    if (err != cudaSuccess)
        return err;
    return cudaMemcpyToSymbol(g_grouped_errors, &zero, sizeof(uint32_t));
}

}  // namespace kvc
