// kvc_grouped.cu -- decode for groups of sequences that share a prefix of pages.
//
// What it computes: the same attention as kvc_decode ("KV Cache Management and
// PagedAttention", "Compute attention over scattered KV"), for sequences whose block tables
// begin with the same physical pages ("Share common KV across responses"; Quail "KV",
// "Prefix sharing").  Each response still attends with its own query over its own context;
// only the reading of the shared pages is done once per group instead of once per member.
//
// Decomposition (all partials are normalised fp32 pieces with their log-sum-exp):
//   setup   grouped_setup_kernel (one block): each sequence's key start (the end of its
//           group's prefix, whole pages; 0 outside groups);
//   prefix  one CTA per (prefix chunk, kv head, group): the chunk's pages, read once, against
//           the query rows of every member of the group (members x G rows, at most 64), on
//           mma.sync tiles of 16 rows;
//   suffix  one decode CTA (kvc_decode_cta.cuh) per (split, kv head, member) over the
//           member's positions from its key start;
//   merge   log-sum-exp over prefix and suffix partials (merge_kernel).
// Prefix and suffix CTAs are one grid (grouped_decode_kernel), prefix CTAs first: the suffix
// CTAs take the SMs as the prefix CTAs drain.  A prefix split that holds no position of its
// group marks the split empty (lse -inf) for the group's rows, and the first suffix CTA of a
// sequence that starts at position 0 (no shared prefix) marks all of its rows' prefix splits
// empty, so every prefix partial the merge reads is written in this grid.  Prefix CTAs read
// nothing the setup kernel writes, so they start without waiting for it (the setup kernel
// itself waits for all earlier work before it lets them launch); suffix CTAs wait for it.  A TMA producer warp streams the prefix pages
// (one box per page) into a 3-deep swizzled ring; four consumer warps cover 1, 2 or 4 row
// tiles, the warps of one tile splitting each 64-position stage between them and combining
// through shared memory at the end.
#include <math.h>

#include "kvc_decode_cta.cuh"
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
    static constexpr int kCombineBytes =
        kConsumerWarps * 16 * (D + 8) * 4 + 2 * kConsumerWarps * 16 * 4 +
        kMaxRows * kConsumerWarps * 4 + kMaxRows * 8;
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
    int chunk, n_split, split_stride;
    float scale_log2;
    int hnd;   // HND pools: page boxes addressed by (page, kv head) block
    int n_items;   // prefix work items: n_split * kv_heads * groups
    uint32_t *err;   // the caller's device error word, or null (this file's own word)
};

// Every sequence's key start: 0, then, for each group member, the end of the group's prefix in
// whole pages (the two phases separated by the block barrier).  One block.
__global__ void grouped_setup_kernel(int32_t *__restrict__ key_start,
                                     const int32_t *__restrict__ group_indptr,
                                     const int32_t *__restrict__ group_seqs,
                                     const int32_t *__restrict__ prefix_len, int num_groups,
                                     int num_seqs, int page_size, int bt_stride)
{
    pdl_wait();
    pdl_trigger();
    for (int s = threadIdx.x; s < num_seqs; s += blockDim.x)
        key_start[s] = 0;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int g = warp; g < num_groups; g += blockDim.x >> 5) {
        int pre = (prefix_len[g] / page_size) * page_size;   // whole pages only
        pre = min(max(pre, 0), bt_stride * page_size);
        for (int i = group_indptr[g] + lane; i < group_indptr[g + 1]; i += 32)
            key_start[group_seqs[i]] = pre;
    }
}

// ------------------------------- group detection --------------------------------------
// Groups from the block tables alone: adjacent sequences s - 1, s are linked when their
// tables agree on at least the first page that both can share (pages wholly before the page
// of the last position); a group is a maximal run of linked sequences cut into chunks of at
// most max_members, chunks of one sequence dropped; its prefix is the smallest agreement
// inside the chunk.  group_agree_kernel measures every adjacent pair's agreement (a warp per
// pair, 32 table entries per step) into group_seqs, which serves as scratch; then one CTA of
// kDetectThreads threads walks the sequences in tiles of kDetectTile, reading a tile's
// agreements (and the next max_members ones) before it writes any output.  Its writes to
// group_seqs land at member offsets <= the sequence index, below every agreement a later
// tile still has to read.
constexpr int kDetectThreads = 1024;
constexpr int kDetectTile = kDetectThreads;
constexpr int kDetectMaxMembers = 64;

// The first kAgreeSpan entries of both rows are requested together with the two context
// lengths (entries below bt_stride are always in the rows), so a pair whose agreement ends
// within them costs one memory round trip; longer agreements go on kAgreeSpan at a time.
constexpr int kAgreeSpan = 128;

__device__ int pair_agreement(const int32_t *__restrict__ bt, int bt_stride,
                              const int32_t *__restrict__ ctx, int page_size, int s, int lane)
{
    if (s == 0)
        return 0;
    constexpr int kPer = kAgreeSpan / 32;
    const int32_t *a = bt + static_cast<size_t>(s - 1) * bt_stride;
    const int32_t *b = bt + static_cast<size_t>(s) * bt_stride;
    int av[kPer], bv[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int k = 32 * u + lane;
        av[u] = k < bt_stride ? a[k] : 0;
        bv[u] = k < bt_stride ? b[k] : 0;
    }
    const int sh0 = min(max(ctx[s - 1] - 1, 0) / page_size, bt_stride);
    const int sh1 = min(max(ctx[s] - 1, 0) / page_size, bt_stride);
    const int lim = min(sh0, sh1);
    for (int k0 = 0; k0 < lim; k0 += kAgreeSpan) {
        if (k0 > 0) {
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int k = k0 + 32 * u + lane;
                av[u] = k < lim ? a[k] : 0;
                bv[u] = k < lim ? b[k] : 0;
            }
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int k = k0 + 32 * u + lane;
            const unsigned diff = __ballot_sync(0xffffffffu, k < lim && av[u] != bv[u]);
            if (diff != 0u)
                return k0 + 32 * u + __ffs(diff) - 1;
        }
    }
    return lim;
}

// Inclusive max / exclusive sum over the block (all kDetectThreads threads call them).
__device__ int block_max_scan(int v, int *red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off)
            v = max(v, o);
    }
    if (lane == 31)
        red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = red[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off)
                w = max(w, o);
        }
        red[lane] = w;
    }
    __syncthreads();
    const int r = warp > 0 ? max(v, red[warp - 1]) : v;
    __syncthreads();
    return r;
}

__device__ int block_sum_scan_excl(int v, int *red, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off)
            x += o;
    }
    if (lane == 31)
        red[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = red[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off)
                w += o;
        }
        red[lane] = w;
    }
    __syncthreads();
    const int r = x - v + (warp > 0 ? red[warp - 1] : 0);
    *total = red[31];
    __syncthreads();
    return r;
}

constexpr int kAgreeWarps = 8;

__global__ void __launch_bounds__(kAgreeWarps * 32)
    group_agree_kernel(const int32_t *__restrict__ bt, int bt_stride,
                       const int32_t *__restrict__ ctx, int num_seqs, int page_size,
                       int32_t *__restrict__ agree_out)
{
    pdl_wait();
    pdl_trigger();
    const int s = blockIdx.x * kAgreeWarps + (threadIdx.x >> 5);
    if (s >= num_seqs)
        return;   // warp-uniform
    const int k = pair_agreement(bt, bt_stride, ctx, page_size, s, threadIdx.x & 31);
    if ((threadIdx.x & 31) == 0)
        agree_out[s] = k;
}

__global__ void __launch_bounds__(kDetectThreads, 1)
    group_detect_kernel(int num_seqs, int page_size, int max_members, int capacity,
                        int32_t *__restrict__ group_indptr, int32_t *group_seqs,
                        int32_t *__restrict__ prefix_len, int32_t *__restrict__ num_groups)
{
    pdl_wait();
    pdl_trigger();
    // agreement of sequences t0 .. t0 + kDetectTile + max_members - 1 of the current tile: a
    // chunk starting in the tile reads its members' agreements past the tile's end
    __shared__ int agree[kDetectTile + kDetectMaxMembers];
    __shared__ int red[32];
    const int tid = threadIdx.x;
    int carry_run = 0, carry_members = 0, carry_groups = 0;
    for (int t0 = 0; t0 < num_seqs; t0 += kDetectTile) {
        const int n_ext = min(kDetectTile + max_members, num_seqs - t0);
        for (int i = tid; i < n_ext; i += kDetectThreads)
            agree[i] = group_seqs[t0 + i];   // the agreements group_agree_kernel left here
        __syncthreads();
        const int s = t0 + tid;
        const bool valid = s < num_seqs;
        // the start of s's run: the last r <= s that is 0 or not linked to r - 1
        const int run = max(block_max_scan(valid && (s == 0 || agree[tid] == 0) ? s : -1, red),
                            carry_run);
        const bool chunk_start = valid && (s - run) % max_members == 0;
        // s is in a group unless it starts a chunk that the next sequence does not continue
        const bool continued =
            s + 1 < num_seqs && tid + 1 < n_ext && agree[tid + 1] >= 1 && max_members >= 2;
        const bool in_group = valid && (!chunk_start || continued);
        const bool group_start = chunk_start && in_group;
        int members_here, groups_here;
        const int mi = carry_members + block_sum_scan_excl(in_group ? 1 : 0, red, &members_here);
        const int gi = carry_groups + block_sum_scan_excl(group_start ? 1 : 0, red, &groups_here);
        if (in_group)
            group_seqs[mi] = s;
        if (group_start && gi < capacity) {
            int pre = agree[tid + 1];
            for (int j = 2; j < max_members && s + j < num_seqs && agree[tid + j] >= 1; ++j)
                pre = min(pre, agree[tid + j]);
            group_indptr[gi] = mi;
            prefix_len[gi] = pre * page_size;
        }
        // the run reaching into the next tile starts where the tile's last sequence's run does
        if (tid == min(kDetectTile, num_seqs - t0) - 1)
            red[0] = run;
        __syncthreads();
        carry_run = red[0];
        carry_members += members_here;
        carry_groups += groups_here;
        __syncthreads();
    }
    // unused group slots: no members, no prefix (a decode over them does nothing); the end
    // offset of the last group and of every unused slot, up to group_indptr[capacity]
    for (int g = min(carry_groups, capacity) + tid; g <= capacity; g += kDetectThreads) {
        group_indptr[g] = carry_members;
        if (g < capacity)
            prefix_len[g] = 0;
    }
    if (tid == 0)
        *num_groups = carry_groups;
}

// One prefix work item: chunk `split` of the shared prefix of group `grp`, kv head `kvh`.
// Returns false in a thread whose bounded wait gave up (its error bit is set).
template <int D, int NMT>
__device__ __forceinline__ bool prefix_cta(const CUtensorMap *tmap_k, const CUtensorMap *tmap_v,
                                           const Args &a, const int split, const int kvh,
                                           const int grp, uint8_t *smem)
{
    using Geom = GroupGeom<D>;
    constexpr int kWarpsPerTile = kConsumerWarps / NMT;   // warps sharing one 16-row tile
    constexpr int kKeysPerWarp = kStageKeys / kWarpsPerTile;
    constexpr int kNT = kKeysPerWarp / 8;                  // n-tiles of S per warp and stage

    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Geom::kRingBytes);
    uint64_t *empty = full + kStages;

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
    if (k_begin >= k_end || rows <= 0) {
        // no position of the group's prefix in this split: empty for each member row
        for (int r = threadIdx.x; r < rows; r += blockDim.x) {
            const int seq = a.group_seqs[m0 + r / G];
            const size_t row = static_cast<size_t>(seq) * a.q_heads +
                               static_cast<size_t>(kvh) * G + (r - (r / G) * G);
            a.part_lse[row * a.split_stride + split] = -INFINITY;
        }
        return true;
    }
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
            prefetch_tensormap(tmap_k);
            prefetch_tensormap(tmap_v);
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
                    tma_load_4d_hint(vdst + off, tmap_v, 0, c1, 0, c3, &full[st], policy);
                else
                    tma_load_4d_hint(kdst + off, tmap_k, 0, c1, 0, c3, &full[st], policy);
            }
            issued = b + 1;
        }
        if (!ok && lane == 0) {
            atomicOr(a.err ? a.err : &g_grouped_errors, kErrDecodeEmptyWait);
            for (int b = max(0, issued - kStages); b < issued; ++b)
                if (!mbar_wait(&full[b % kStages], (b / kStages) & 1))
                    atomicOr(a.err ? a.err : &g_grouped_errors, kErrDrainWait);
        }
        return ok;
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
    float m_a = -INFINITY, m_b = -INFINITY;

    // ldmatrix addresses.  Inside a stage tile, row `row` of half `h` starts at
    // ((row / P) * (D / 64) + h) * P * 128 + (row % P) * 128, and 16-byte chunk c of it sits
    // at chunk c ^ (row & 7).  Every row a lane addresses has row & 7 equal to lane & 7, so the
    // swizzled chunk of column tile j is (2 (j % 4) + c0) ^ (lane & 7), i.e. (32 (j % 4)) ^ x
    // bytes for a per-lane x: one add per ldmatrix once the row's offset is known.
    const int log2p = __ffs(P) - 1;
    const int half_bytes = P * 128;
    constexpr int kHalves = D / 64;
    constexpr int kPairs = kNT / 2;             // 16-key groups of a warp's slice
    const int k_row = ksl * kKeysPerWarp + (lane & 7) + ((lane >> 4) << 3);
    const int v_row = ksl * kKeysPerWarp + (lane & 7) + (((lane >> 3) & 1) << 3);
    auto row_offset = [&](int row) {
        return static_cast<uint32_t>(((row >> log2p) * kHalves) * half_bytes +
                                     (row & (P - 1)) * 128);
    };
    uint32_t k_x[4], v_x[4];
    {
        const uint32_t xk = static_cast<uint32_t>((((lane >> 3) & 1) ^ (lane & 7)) << 4);
        const uint32_t xv = static_cast<uint32_t>(((lane >> 4) ^ (lane & 7)) << 4);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            k_x[j] = (32u * j) ^ xk;
            v_x[j] = (32u * j) ^ xv;
        }
    }
    // Row sums of the bf16 probabilities come out of the P.V products: one more n-tile
    // whose B operand is all ones sums P's rows exactly as the products see them.
    constexpr uint32_t kOnes = 0x3F803F80u;   // two bf16 1.0
    float o_l[4] = {0.0f, 0.0f, 0.0f, 0.0f};
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
            for (int pr = 0; pr < kPairs; ++pr) {
                const uint32_t krow = kbase + row_offset(pr * 16 + k_row);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(krow + (kk / 4) * half_bytes + k_x[kk % 4], b0, b1, b2, b3);
                    mma_bf16_16816(sc[2 * pr], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0,
                                   b1);
                    mma_bf16_16816(sc[2 * pr + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3],
                                   b2, b3);
                }
            }
            if (n_valid < kKeysPerWarp) {   // warp-uniform: only the last slice of a chunk
#pragma unroll
                for (int n = 0; n < kNT; ++n) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        if (n * 8 + cq + e >= n_valid) {
                            sc[n][e] = -INFINITY;
                            sc[n][2 + e] = -INFINITY;
                        }
                    }
                }
            }
            float mx_a = fmax3(sc[0][0], sc[0][1], sc[1][0]);
            float mx_b = fmax3(sc[0][2], sc[0][3], sc[1][2]);
            mx_a = fmaxf(mx_a, sc[1][1]);
            mx_b = fmaxf(mx_b, sc[1][3]);
#pragma unroll
            for (int n = 2; n < kNT; ++n) {
                mx_a = fmax3(mx_a, sc[n][0], sc[n][1]);
                mx_b = fmax3(mx_b, sc[n][2], sc[n][3]);
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
                o_l[0] *= al_a;
                o_l[1] *= al_a;
                o_l[2] *= al_b;
                o_l[3] *= al_b;
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
            }
#pragma unroll
            for (int ks = 0; ks < kPairs; ++ks) {
                if (ks * 16 >= n_valid)
                    break;
                const bool partial = n_valid < (ks + 1) * 16;
                const uint32_t vrow = vbase + row_offset(ks * 16 + v_row);
#pragma unroll
                for (int dt = 0; dt < D / 16; ++dt) {
                    uint32_t v0, v1, v2, v3;
                    ldsm_x4_trans(vrow + (dt / 4) * half_bytes + v_x[dt % 4], v0, v1, v2, v3);
                    if (partial) {
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
                mma_bf16_16816(o_l, pa[2 * ks][0], pa[2 * ks][1], pa[2 * ks + 1][0],
                               pa[2 * ks + 1][1], kOnes, kOnes);
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[st]);
    }
    if (!ok)
        atomicOr(a.err ? a.err : &g_grouped_errors, kErrDecodeFullWait);

    // ------------------- combine the warps of each tile, write partials --------------------
    // Warp w of tile t leaves its unnormalised o (rows of D + 8 floats: the pad spreads the
    // 8 rows a store instruction touches over distinct banks), its running max and row sum.
    // One thread per output row then folds the tile's warps into weights 2^(m_w - M) / L
    // and finds the row's partial slot; the write-out is float4 loads and stores.
    constexpr int kRowStride = D + 8;
    const float l_a = o_l[0], l_b = o_l[2];   // every column of the ones tile holds the sum
    named_barrier(1, kConsumerWarps * 32);   // every warp is done with the ring
    float *red_o = reinterpret_cast<float *>(smem);                        // [W][16][D + 8]
    float *red_m = red_o + kConsumerWarps * 16 * kRowStride;                // [W][16]
    float *red_l = red_m + kConsumerWarps * 16;                             // [W][16]
    float *row_w = red_l + kConsumerWarps * 16;                             // [rows][W / tile]
    long long *row_slot = reinterpret_cast<long long *>(row_w + kMaxRows * kWarpsPerTile);
    {
        const int la = lane >> 2, lb = la + 8;
        float *dst_a = red_o + (warp * 16 + la) * kRowStride + cq;
        float *dst_b = red_o + (warp * 16 + lb) * kRowStride + cq;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            *reinterpret_cast<float2 *>(dst_a + n * 8) = make_float2(o[n][0], o[n][1]);
            *reinterpret_cast<float2 *>(dst_b + n * 8) = make_float2(o[n][2], o[n][3]);
        }
        if ((lane & 3) == 0) {
            red_m[warp * 16 + la] = m_a;
            red_l[warp * 16 + la] = l_a;
            red_m[warp * 16 + lb] = m_b;
            red_l[warp * 16 + lb] = l_b;
        }
    }
    named_barrier(1, kConsumerWarps * 32);
    for (int r = threadIdx.x; r < rows; r += kConsumerWarps * 32) {
        const int slot0 = (r >> 4) * kWarpsPerTile * 16 + (r & 15);
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarpsPerTile; ++w)
            M = fmaxf(M, red_m[slot0 + w * 16]);
        float f[kWarpsPerTile];
        float L = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarpsPerTile; ++w) {
            const float mw = red_m[slot0 + w * 16];
            f[w] = (mw == -INFINITY) ? 0.0f : fast_exp2(mw - M);
            L += f[w] * red_l[slot0 + w * 16];
        }
        const float inv = (L > 0.0f) ? 1.0f / L : 0.0f;
#pragma unroll
        for (int w = 0; w < kWarpsPerTile; ++w)
            row_w[r * kWarpsPerTile + w] = f[w] * inv;
        const int m = r / G;
        const int gh = r - m * G;
        const int seq = a.group_seqs[m0 + m];
        const long long prow =
            (static_cast<long long>(seq) * a.q_heads + static_cast<long long>(kvh) * G + gh) *
                a.split_stride + split;
        row_slot[r] = prow;
        a.part_lse[prow] = (L > 0.0f) ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
    named_barrier(1, kConsumerWarps * 32);
    constexpr int kVec = D / 4;
    for (int idx = threadIdx.x; idx < rows * kVec; idx += kConsumerWarps * 32) {
        const int r = idx / kVec;
        const int c = (idx - r * kVec) * 4;
        const float *src = red_o + ((r >> 4) * kWarpsPerTile * 16 + (r & 15)) * kRowStride + c;
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int w = 0; w < kWarpsPerTile; ++w) {
            const float wt = row_w[r * kWarpsPerTile + w];
            const float4 v = *reinterpret_cast<const float4 *>(src + w * 16 * kRowStride);
            acc.x = fmaf(wt, v.x, acc.x);
            acc.y = fmaf(wt, v.y, acc.y);
            acc.z = fmaf(wt, v.z, acc.z);
            acc.w = fmaf(wt, v.w, acc.w);
        }
        *reinterpret_cast<float4 *>(a.part_o + row_slot[r] * D + c) = acc;
    }
    return ok;
}

// The whole shared-prefix decode in one grid: CTAs [0, n_prefix) are prefix CTAs ordered
// (split, kv head, group), the rest the members' suffix decode ordered (split, kv head,
// sequence).  CTAs start roughly in index order, so the suffix CTAs fill the SMs as the prefix
// CTAs drain instead of waiting for the last of them.
template <int D, int NMT>
__global__ void __launch_bounds__(kThreads, 2)
    grouped_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, const Args a,
                          const dec::Args da, const int n_prefix_ctas)
{
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int idx = blockIdx.x;
    if (idx < n_prefix_ctas) {
        // reads only inputs older than the setup kernel (queries, tables, groups), which has
        // itself waited for all earlier work before letting this grid launch.
        // Work items idx, idx + n_prefix_ctas, ... (at most one resident wave of prefix CTAs):
        // the first is taken as it comes; the others are checked for members 32 at a time in
        // one read, so that a group list with empty slots (device-found groups fill a fixed
        // capacity) costs a load per slot, not a CTA.  An item with members but no prefix
        // position in its split still runs: it writes its rows' empty partials.
        const int lane = threadIdx.x & 31;
        int it = idx;
        int batch = idx;                     // todo bit k: item batch + k * n_prefix_ctas
        int next = idx + n_prefix_ctas;      // the first item not yet checked
        uint32_t todo = 0u;
        for (;;) {
            const int split = it % a.n_split;
            const int rest = it / a.n_split;
            const bool ok = prefix_cta<D, NMT>(&tmap_k, &tmap_v, a, split, rest % a.kv_heads,
                                               rest / a.kv_heads, smem);
            while (todo == 0u && next < a.n_items) {
                const long long c = next + static_cast<long long>(lane) * n_prefix_ctas;
                bool live = false;
                if (c < a.n_items) {
                    const int grp = static_cast<int>(c / a.n_split) / a.kv_heads;
                    live = a.group_indptr[grp + 1] > a.group_indptr[grp];
                }
                todo = __ballot_sync(0xffffffffu, live);
                batch = next;
                next += 32 * n_prefix_ctas;
            }
            if (todo == 0u)
                break;
            // the item is done with the ring, the barriers and the combine's shared memory
            // before the next one's bulk copies write there; stop after a failed wait
            fence_proxy_async_smem();
            if (__syncthreads_or(!ok))
                break;
            it = batch + (__ffs(todo) - 1) * n_prefix_ctas;
            todo &= todo - 1u;
        }
    } else {
        pdl_wait();   // the key starts
        const int j = idx - n_prefix_ctas;
        const int split = j % da.n_split;
        const int rest = j / da.n_split;
        const int kvh = rest % da.kv_heads;
        const int s = rest / da.kv_heads;
        if (split == 0 && da.key_start[s] == 0) {
            // a sequence without a shared prefix: its rows' prefix splits are empty
            const int G = da.group;
            for (int t = threadIdx.x; t < G * a.n_split; t += blockDim.x) {
                const size_t row = static_cast<size_t>(s) * da.q_heads +
                                   static_cast<size_t>(kvh) * G + t / a.n_split;
                a.part_lse[row * a.split_stride + (t - (t / a.n_split) * a.n_split)] = -INFINITY;
            }
        }
        dec::decode_cta<D, true>(&tmap_k, &tmap_v, da, split, kvh, s, smem,
                                 da.err ? da.err : &g_grouped_errors);
    }
}

template <int D, int NMT>
cudaError_t launch_t(const GroupedPrefixLaunch &p, const DecodeLaunch &l, const CUtensorMap &tk,
                     const CUtensorMap &tv, cudaStream_t stream)
{
    static_assert(kThreads == dec::kThreads, "prefix and suffix CTAs share the block shape");
    Args a;
    a.q = static_cast<const __nv_bfloat16 *>(p.q);
    a.part_o = p.part_o;
    a.part_lse = p.part_lse;
    a.block_table = p.block_table;
    a.bt_stride = p.bt_stride;
    a.group_indptr = p.group_indptr;
    a.group_seqs = p.group_seqs;
    a.prefix_len = p.prefix_len;
    a.q_heads = p.q_heads;
    a.kv_heads = p.kv_heads;
    a.hnd = p.hnd ? 1 : 0;
    a.err = current_error_word();
    a.group = p.q_heads / p.kv_heads;
    a.page_size = p.page_size;
    a.chunk = p.chunk;
    a.n_split = p.n_split > 0 ? p.n_split : 1;
    a.split_stride = p.split_stride;
    a.scale_log2 = p.scale * kLog2e;
    const dec::Args da = dec::make_args(l);
    const long long n_items =
        p.num_groups > 0 ? static_cast<long long>(p.n_split) * p.kv_heads * p.num_groups : 0;
    if (n_items > 0x3FFFFFFFLL)
        return cudaErrorInvalidConfiguration;
    a.n_items = static_cast<int>(n_items);
    const long long n_prefix =
        p.max_prefix_ctas > 0 && n_items > p.max_prefix_ctas ? p.max_prefix_ctas : n_items;
    const long long n_ctas =
        n_prefix + static_cast<long long>(l.n_split) * l.kv_heads * l.num_seqs;
    if (n_ctas == 0)
        return cudaSuccess;
    if (n_ctas > 0x7FFFFFFFLL)
        return cudaErrorInvalidConfiguration;
    const size_t smem = GroupGeom<D>::kSmemBytes > dec::DecodeGeom<D>::kSmemBytes
                            ? GroupGeom<D>::kSmemBytes
                            : dec::DecodeGeom<D>::kSmemBytes;
    auto kernel = grouped_decode_kernel<D, NMT>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess)
        return err;
    return launch_pdl(kernel, dim3(static_cast<unsigned>(n_ctas)), dim3(kThreads), smem, stream,
                      tk, tv, a, da, static_cast<int>(n_prefix));
}

template <int D>
cudaError_t launch_d(const GroupedPrefixLaunch &p, const DecodeLaunch &l, const CUtensorMap &tk,
                     const CUtensorMap &tv, cudaStream_t stream)
{
    if (p.max_rows <= 16)
        return launch_t<D, 1>(p, l, tk, tv, stream);
    if (p.max_rows <= 32)
        return launch_t<D, 2>(p, l, tk, tv, stream);
    return launch_t<D, 4>(p, l, tk, tv, stream);
}

}  // namespace

cudaError_t launch_grouped_setup(int32_t *key_start, const int32_t *group_indptr,
                                 const int32_t *group_seqs, const int32_t *prefix_len,
                                 int num_groups, int num_seqs, int page_size, int bt_stride,
                                 cudaStream_t stream)
{
    return launch_pdl(grouped_setup_kernel, dim3(1), dim3(256), 0, stream, key_start,
                      group_indptr, group_seqs, prefix_len, num_groups, num_seqs, page_size,
                      bt_stride);
}

cudaError_t launch_group_detect(const int32_t *block_table, int bt_stride,
                                const int32_t *context_lens, int num_seqs, int page_size,
                                int max_members, int32_t *group_indptr, int32_t *group_seqs,
                                int32_t *prefix_len, int32_t *num_groups, cudaStream_t stream)
{
    if (max_members < 2 || max_members > kDetectMaxMembers)
        return cudaErrorInvalidValue;
    if (num_seqs > 0) {
        const cudaError_t err = launch_pdl(
            group_agree_kernel, dim3((num_seqs + kAgreeWarps - 1) / kAgreeWarps),
            dim3(kAgreeWarps * 32), 0, stream, block_table, bt_stride, context_lens, num_seqs,
            page_size, group_seqs);
        if (err != cudaSuccess)
            return err;
    }
    return launch_pdl(group_detect_kernel, dim3(1), dim3(kDetectThreads), 0, stream, num_seqs,
                      page_size, max_members, num_seqs / 2, group_indptr, group_seqs,
                      prefix_len, num_groups);
}

cudaError_t launch_grouped_decode(const GroupedPrefixLaunch &p, const DecodeLaunch &l,
                                  const CUtensorMap &tk, const CUtensorMap &tv,
                                  cudaStream_t stream)
{
    return p.head_dim == 128 ? launch_d<128>(p, l, tk, tv, stream)
                             : launch_d<64>(p, l, tk, tv, stream);
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
