// kvc_decode_int8.cu -- paged decode attention over INT8 pages.
//
// What it computes: the attention of kvc_decode ("KV Cache Management and PagedAttention",
// "Compute attention over scattered KV") over pages that hold int8 codes with one fp32 scale
// per (position, kv head) vector (TileInfer.jl "KV cache", "INT8 cache").  As that section
// says, the cache is not dequantised: a key's scale multiplies its score, and a value's scale
// its probability before the PV product.  Codes are converted to fp16 in registers (exact:
// |code| <= 127) for the tensor cores; the scales stay outside the products.  fp16 rather than
// bf16 because two codes become an exact fp16 pair in three integer/half operations: bytes
// b placed under the exponent 0x64 read as 1024 + b, and the code is b - 128; the query is
// converted to fp16 once (scaled by a power of two when it would overflow fp16), and the
// probabilities (at most 1) times the value scales enter the PV product as fp16.
//
// Layout: codes [num_pages * P][Hkv][128] int8 like the bf16 pools (128 bytes per vector);
// scales [num_pages][Hkv][P] fp32, so the P scales of one (page, kv head) are one contiguous
// run that a single bulk copy brings in.
//
// Kernel design (head_dim 128): one CTA per (split, kv head, sequence), 4 consumer warps and a
// producer warp, three CTAs per SM.  The producer streams 64-position stages -- per page one TMA
// box of K codes, one of V codes (128-byte swizzle) and one bulk copy each of the K and V
// scales, issued by parallel lanes -- through a 4-deep ring.  Consumer warp w takes positions
// 16 w .. 16 w + 15 of each stage:
//   S = Q K^T on mma.sync m16n8k16 (fp16; the G query heads padded to 16 rows).  The order
//   in which head_dim is contracted is free, so thread (., t) takes dims 32 t + 4 kk .. + 3
//   for k-step kk: its K codes for a position are 32 contiguous bytes (two 16-byte loads) and
//   its Q pairs two contiguous pairs;
//   O^T += V^T (P * v_scale)^T with M = 16 dims and N = 8 query rows: the probabilities a
//   thread holds from the S fragment are exactly its B fragment, half as many MMAs and
//   accumulators as O = P V with rows padded to 16; the dims of tile dt are permuted so that
//   thread row r reads dims 32 q + 4 r .. + 3 (q = 0..3), one 4-byte word per position and q,
//   and the accumulators are put back in dim order when the warps combine.
// Online softmax in base 2, masked positions excluded before the exponential and their
// probabilities set to 0 by selection (a scale left in an unused slot may be NaN).
// Fused store (kvc_decode_int8_store): the producer of the CTA whose chunk ends at a
// sequence's newest position quantises that token's K/V row with the INT8 store's arithmetic
// and writes its codes and scale before the copies of that page.
#include <math.h>

#include "kvc_device.cuh"
#include "kvc_launch.h"

namespace kvc {

namespace {

__device__ uint32_t g_decode_int8_errors;

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 4;
constexpr int kKeysPerWarp = kStageKeys / kConsumerWarps;   // 16
constexpr int kMaxGroup = 8;
constexpr float kLn2 = 0.6931471805599453f;

// Stage layout for head_dim D (64 or 128): K codes [64 rows][D], V codes, K scales, V scales.
template <int D>
struct I8Geom {
    static constexpr int kCodeBytes = kStageKeys * D;        // K (or V) codes of one stage
    static constexpr int kScaleBytes = kStageKeys * 4;
    static constexpr int kOffV = kCodeBytes;
    static constexpr int kOffKs = 2 * kCodeBytes;
    static constexpr int kOffVs = kOffKs + kScaleBytes;
    static constexpr int kStageBytes = ((2 * kCodeBytes + 2 * kScaleBytes) + 1023) & ~1023;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kCombineBytes =   // o rows, m, l per warp; weights per row
        kConsumerWarps * kMaxGroup * (D + 4) * 4 + 3 * kConsumerWarps * kMaxGroup * 4;
    static_assert(kCombineBytes <= kRingBytes, "combine area aliases the ring");
    static constexpr size_t kSmemBytes = 1024 + kRingBytes + 2 * kStages * 8;
};

struct Args {
    const __nv_bfloat16 *q;
    const float *k_scales, *v_scales;
    void *out;
    int out_f32;
    float *part_o;
    float *part_lse;
    const int32_t *block_table;
    int bt_stride;
    const int32_t *context_lens;
    int q_heads, kv_heads, group, page_size;
    int chunk, n_split;
    float scale_log2;
    // kvc_decode_int8_store: sequence s's new key and value (bf16 [S][Hkv][D]), quantised and
    // written to the code and scale pools (num_slots slots) by the CTA whose chunk ends at the
    // newest position, before that CTA's copies of the page; null otherwise.
    const __nv_bfloat16 *k_new, *v_new;
    int8_t *k_codes_w, *v_codes_w;
    float *k_scales_w, *v_scales_w;
    int num_slots;
    uint32_t *err;   // the caller's device error word, or null (this file's own word)
    int hnd;         // HND codes: page boxes addressed by (offset, page * kv_heads + kv head)
};

// Quantises one vector held as E bf16 values per lane (lane l: elements E l .. E l + E - 1;
// E = head_dim / 32, packed two per word) and writes its codes and scale, with the arithmetic
// of kvc_store_int8 (TileInfer.jl "KV cache", "INT8 cache": scale = max |x| / 127, codes
// rounded to nearest and clamped to +-127, both quotients fp32 round-to-nearest), so both give
// the same bytes.
template <int E>
__device__ __forceinline__ void quantise_store_row(const uint32_t (&x)[E / 2], int8_t *codes,
                                                   float *scale_out, int lane)
{
    float f[E];
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
        f[2 * i] = __uint_as_float(x[i] << 16);
        f[2 * i + 1] = __uint_as_float(x[i] & 0xFFFF0000u);
    }
    float m = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e)
        m = fmaxf(m, fabsf(f[e]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const float scale = __fdiv_rn(m, 127.0f);
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        int c = 0;
        if (scale != 0.0f)
            c = max(-127, min(127, __float2int_rn(__fdiv_rn(f[e], scale))));
        packed |= (static_cast<uint32_t>(c) & 0xFFu) << (8 * e);
    }
    if (E == 4)
        *reinterpret_cast<uint32_t *>(codes + lane * 4) = packed;
    else
        *reinterpret_cast<uint16_t *>(codes + lane * 2) = static_cast<uint16_t>(packed);
    if (lane == 0)
        *scale_out = scale;
}

// fp16 pair (low: byte c of a, high: byte c of b) of two words of int8 codes, exact.  The
// bytes are moved under exponent bits 0x64 (fp16 1024 + m for m in 0..255) with the sign bit
// of the code flipped (m = code + 128), and 1152 is subtracted from both halves.
template <int c>
__device__ __forceinline__ uint32_t codes_f16x2(uint32_t a, uint32_t b)
{
    const uint32_t bytes = __byte_perm(a, b, c | ((4 + c) << 8));   // [a.c, a.0, b.c, a.0]
    const uint32_t biased = (bytes & 0x00FF00FFu) ^ 0x64806480u;
    const __half2 h = __hsub2(*reinterpret_cast<const __half2 *>(&biased),
                              __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Offset of byte `col` of stage row `row` in a [64][D] code tile: 128-byte rows with the
// 128-byte swizzle (16-byte chunk c of row r at c ^ (r % 8)), or 64-byte rows with the 64-byte
// swizzle (chunk c of row r at c ^ ((r / 2) % 4)).
template <int D>
__device__ __forceinline__ uint32_t code_offset(int row, int col)
{
    const int phase = D == 128 ? (row & 7) : ((row >> 1) & 3);
    return static_cast<uint32_t>(row * D + ((((col >> 4) ^ phase)) << 4) + (col & 15));
}

template <int D, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 3)
    paged_decode_int8_kernel(const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v, const Args a)
{
    pdl_wait();
    pdl_trigger();
    using Geom = I8Geom<D>;
    constexpr int kOffV = Geom::kOffV, kOffKs = Geom::kOffKs, kOffVs = Geom::kOffVs;
    constexpr int kStageBytes = Geom::kStageBytes, kRingBytes = Geom::kRingBytes;
    constexpr int E = D / 32;   // values of one vector per lane (the fused store)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kRingBytes);
    uint64_t *empty = full + kStages;

    const int split = blockIdx.x;
    const int kvh = blockIdx.y;
    const int s = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.group;
    const int P = a.page_size;
    // the new token's row, requested before anything else so that it is in registers by the
    // time the producer writes it
    uint32_t k_row_new[E / 2] = {}, v_row_new[E / 2] = {};
    if (a.k_new != nullptr && warp == kConsumerWarps) {
        const size_t src = ((static_cast<size_t>(s) * a.kv_heads + kvh) * 32 + lane) * (E / 2);
        const uint32_t *kn = reinterpret_cast<const uint32_t *>(a.k_new) + src;
        const uint32_t *vn = reinterpret_cast<const uint32_t *>(a.v_new) + src;
#pragma unroll
        for (int i = 0; i < E / 2; ++i) {
            k_row_new[i] = __ldg(kn + i);
            v_row_new[i] = __ldg(vn + i);
        }
    }
    int ctx = a.context_lens[s];
    bool store_new = a.k_new != nullptr && ctx >= 1;
    if (ctx > a.bt_stride * P) {
        if (threadIdx.x == 0 && split == 0)
            atomicOr(a.err ? a.err : &g_decode_int8_errors, kErrContextRange);
        ctx = a.bt_stride * P;
        store_new = false;   // no slot for the new token: stored nowhere
    }
    const int k_begin = split * a.chunk;
    const int k_end = min(ctx, k_begin + a.chunk);
    const size_t row0 = static_cast<size_t>(s) * a.q_heads + static_cast<size_t>(kvh) * G;

    if (k_begin >= k_end) {
        if (SPLIT) {
            if (threadIdx.x < G)
                a.part_lse[(row0 + threadIdx.x) * a.n_split + split] = -INFINITY;
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
        // ------------------------ producer (whole warp) -------------------------------------
        const int32_t *bt_row =
            a.block_table + static_cast<size_t>(s) * a.bt_stride + first_page;
        if (lane == 0) {
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
        }
        const uint64_t policy = l2_policy_evict_first();
        int cached_base = -32;
        int cached_page = 0;
        int issued = 0;
        bool ok = true;
        // this CTA writes the new token when its chunk ends at the newest position: before
        // the last stage's copies read that page's codes and scales
        const bool writes_new = store_new && k_end == ctx;
        const int new_page = writes_new ? a.block_table[static_cast<size_t>(s) * a.bt_stride +
                                                        (ctx - 1) / P]
                                        : 0;
        for (int b = 0; b < n_blocks; ++b) {
            const int st = b % kStages;
            if (b >= kStages &&
                !__all_sync(0xffffffffu, mbar_wait(&empty[st], ((b / kStages) - 1) & 1))) {
                ok = false;
                break;
            }
            const int rel0 = b * kStageKeys;
            const int keys = min(kStageKeys, k_end - k_begin - rel0);
            const int np = (keys + P - 1) / P;
            if (lane == 0)
                mbar_arrive_expect_tx(&full[st],
                                      static_cast<uint32_t>(np * P * (2 * D + 2 * 4)));
            __syncwarp();
            uint8_t *stage = smem + st * kStageBytes;
            const int lp0 = rel0 / P;
            if (lp0 + np > cached_base + 32) {
                cached_base = lp0;
                cached_page = (lp0 + lane < n_pages) ? bt_row[lp0 + lane] : 0;
            }
            // lane 4 i + op: page i's K codes, V codes, K scales, V scales
            const int i = lane >> 2;
            const int op = lane & 3;
            const int page = __shfl_sync(0xffffffffu, cached_page, (lp0 - cached_base + i) & 31);
            if (writes_new && b + 1 == n_blocks) {
                const int off_new = (ctx - 1) % P;
                const long long slot = static_cast<long long>(new_page) * P + off_new;
                if (new_page >= 0 && slot < a.num_slots) {
                    const size_t sidx =
                        (static_cast<size_t>(new_page) * a.kv_heads + kvh) * P + off_new;
                    const size_t row =
                        (a.hnd ? sidx : static_cast<size_t>(slot) * a.kv_heads + kvh) * D;
                    quantise_store_row<E>(k_row_new, a.k_codes_w + row, a.k_scales_w + sidx,
                                          lane);
                    quantise_store_row<E>(v_row_new, a.v_codes_w + row, a.v_scales_w + sidx,
                                          lane);
                } else if (lane == 0) {
                    atomicOr(a.err ? a.err : &g_decode_int8_errors, kErrSlotRange);   // skipped, as in the store
                }
                // the stores (generic proxy) before the copies (async proxy) that read them
                fence_proxy_async_global();
                __syncwarp();
                fence_proxy_async_global();
            }
            if (i < np) {
                if (op == 0) {
                    tma_load_3d(stage + i * P * D, &tmap_k, 0, a.hnd ? 0 : kvh,
                                a.hnd ? page * a.kv_heads + kvh : page * P, &full[st], policy);
                } else if (op == 1) {
                    tma_load_3d(stage + kOffV + i * P * D, &tmap_v, 0, a.hnd ? 0 : kvh,
                                a.hnd ? page * a.kv_heads + kvh : page * P, &full[st], policy);
                } else {
                    const float *src = (op == 2 ? a.k_scales : a.v_scales) +
                                       (static_cast<size_t>(page) * a.kv_heads + kvh) * P;
                    bulk_load(stage + (op == 2 ? kOffKs : kOffVs) + i * P * 4, src, P * 4,
                              &full[st]);
                }
            }
            issued = b + 1;
        }
        if (!ok && lane == 0) {
            atomicOr(a.err ? a.err : &g_decode_int8_errors, kErrDecodeEmptyWait);
            for (int b = max(0, issued - kStages); b < issued; ++b)
                if (!mbar_wait(&full[b % kStages], (b / kStages) & 1))
                    atomicOr(a.err ? a.err : &g_decode_int8_errors, kErrDrainWait);
        }
        return;
    }

    // --------------------------------- consumers -----------------------------------------
    const int r = lane >> 2;   // fragment row = q head of the group (rows >= G: padding)
    const int t = lane & 3;
    // Q pairs in the contraction order (k-step kk uses dims 32 t + 4 kk + {0, 1} and {2, 3}),
    // as fp16.  A power of two q_pow brings the largest |q| of the group below 2^14 when it
    // is above, and is folded back into the score scale (exact either way).
    uint32_t qa[D / 16][2];
    float sl2 = a.scale_log2;
    {
        const __nv_bfloat16 *qrow = a.q + (row0 + r) * D + (D / 4) * t;
        float qv[D / 4];
        float qmax = 0.0f;
#pragma unroll
        for (int i = 0; i < D / 4; ++i) {
            qv[i] = r < G ? __bfloat162float(qrow[i]) : 0.0f;
            qmax = fmaxf(qmax, fabsf(qv[i]));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, off));
        float q_pow = 1.0f;
        while (qmax * q_pow > 16384.0f)
            q_pow *= 0.5f;
        sl2 = sl2 / q_pow;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qa[kk][0] = pack_f16x2(qv[4 * kk] * q_pow, qv[4 * kk + 1] * q_pow);
            qa[kk][1] = pack_f16x2(qv[4 * kk + 2] * q_pow, qv[4 * kk + 3] * q_pow);
        }
    }
    // O^T accumulators: tile dt holds dims pi(dt, m) x query rows n, this thread rows 2t,
    // 2t + 1 of dims pi(dt, r) (c0, c1) and pi(dt, r + 8) (c2, c3), where
    // pi(dt, r + 8 h) = 32 (dt >> 1) + 4 r + 2 (dt & 1) + h
    float o[D / 16][4];
#pragma unroll
    for (int n = 0; n < D / 16; ++n)
        o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
    float m_run = -INFINITY;
    float l_run = 0.0f;
    const int wrow = warp * kKeysPerWarp;   // first stage row of this warp
    // Stage-independent offsets.  K: the two 16-byte halves of this thread's 32 bytes in rows
    // wrow + r and wrow + 8 + r.  V: the word of dims 4 r .. 4 r + 3 in each of the thread's
    // four positions; dims 32 q + 4 r lie at that offset xor (q << 5), since the swizzle only
    // permutes 16-byte chunks within a row and q moves the chunk index by 2 q.
    constexpr int kKChunks = D / 64;   // 16-byte chunks of this thread's K bytes per row
    uint32_t k_off[2][kKChunks];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int h = 0; h < kKChunks; ++h)
            k_off[nt][h] = code_offset<D>(wrow + 8 * nt + r, (D / 4) * t + 16 * h);
    const int key[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
    uint32_t v_off[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        v_off[i] = kOffV + code_offset<D>(wrow + key[i], 4 * r);
    bool ok = true;

    for (int b = 0; b < n_blocks; ++b) {
        const int st = b % kStages;
        if (!mbar_wait(&full[st], (b / kStages) & 1)) {
            ok = false;
            break;
        }
        const uint8_t *stage = smem + st * kStageBytes;
        const float *ks = reinterpret_cast<const float *>(stage + kOffKs) + wrow;
        const float *vs = reinterpret_cast<const float *>(stage + kOffVs) + wrow;
        const int n_valid = k_end - (k_begin + b * kStageKeys + wrow);
        if (n_valid > 0) {
            // S = Q K^T: B column r of n-tile nt is position 8 nt + r of this warp
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                uint32_t w[D / 16];
#pragma unroll
                for (int h = 0; h < kKChunks; ++h) {
                    const uint4 c4 = *reinterpret_cast<const uint4 *>(stage + k_off[nt][h]);
                    w[4 * h] = c4.x;
                    w[4 * h + 1] = c4.y;
                    w[4 * h + 2] = c4.z;
                    w[4 * h + 3] = c4.w;
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    uint32_t b0, b1;   // codes 0, 1 and codes 2, 3 of the word
                    codes_word_f16x2(w[kk], b0, b1);
                    mma_f16_16816(sc[nt], qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
                }
            }
            // scores of positions 2t, 2t+1 (tile 0) and 8+2t, 9+2t (tile 1), key-scaled
            float x[4] = {sc[0][0], sc[0][1], sc[1][0], sc[1][1]};
#pragma unroll
            for (int i = 0; i < 4; ++i)
                x[i] = key[i] < n_valid ? x[i] * ks[key[i]] * sl2 : -INFINITY;
            float mb = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
            const float m_new = fmaxf(m_run, mb);
            if (__any_sync(0xffffffffu, m_new > m_run)) {
                const float alpha = (m_run == -INFINITY) ? 0.0f : fast_exp2(m_run - m_new);
                // this thread's accumulators are rows 2t and 2t + 1 (held by lanes 8t, 8t + 4)
                const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * t);
                const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * t + 4);
#pragma unroll
                for (int n = 0; n < D / 16; ++n) {
                    o[n][0] *= a0;
                    o[n][1] *= a1;
                    o[n][2] *= a0;
                    o[n][3] *= a1;
                }
                l_run *= alpha;
                m_run = m_new;
            }
            const float m_use = (m_run == -INFINITY) ? 0.0f : m_run;
            float p[4], pv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                p[i] = fast_exp2(x[i] - m_use);
                pv[i] = key[i] < n_valid ? p[i] * vs[key[i]] : 0.0f;
            }
            l_run += (p[0] + p[1]) + (p[2] + p[3]);
            const uint32_t pa0 = pack_f16x2(pv[0], pv[1]);   // positions 2t, 2t+1
            const uint32_t pa2 = pack_f16x2(pv[2], pv[3]);   // positions 8+2t, 9+2t
            // O^T += V^T P'^T: A = V^T (16 dims x 16 positions), B = P'^T, whose fragment is
            // exactly this thread's (pa0, pa2); thread r reads one word (dims 32 q + 4 r .. + 3)
            // of each of its four positions per q
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t vw[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    vw[i] = *reinterpret_cast<const uint32_t *>(stage + (v_off[i] ^ (q << 5)));
                mma_f16_16816(o[2 * q], codes_f16x2<0>(vw[0], vw[1]), codes_f16x2<1>(vw[0], vw[1]),
                              codes_f16x2<0>(vw[2], vw[3]), codes_f16x2<1>(vw[2], vw[3]), pa0,
                              pa2);
                mma_f16_16816(o[2 * q + 1], codes_f16x2<2>(vw[0], vw[1]),
                              codes_f16x2<3>(vw[0], vw[1]), codes_f16x2<2>(vw[2], vw[3]),
                              codes_f16x2<3>(vw[2], vw[3]), pa0, pa2);
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[st]);
    }
    if (!ok)
        atomicOr(a.err ? a.err : &g_decode_int8_errors, kErrDecodeFullWait);

    // ------------------------- combine the 4 warps' partial results -----------------------
    // Each warp leaves its unnormalised o rows (D + 4 floats apart: 16-byte aligned rows),
    // running max and row sum; one thread per query head folds them into weights
    // 2^(m_w - M) / L, and the output is written as float4 (bf16x4) pieces.
    constexpr int kRowStride = D + 4;
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    named_barrier(1, kConsumerWarps * 32);
    float *red_o = reinterpret_cast<float *>(smem);                      // [W][8][D + 4]
    float *red_m = red_o + kConsumerWarps * kMaxGroup * kRowStride;       // [W][8]
    float *red_l = red_m + kConsumerWarps * kMaxGroup;                    // [W][8]
    float *row_w = red_l + kConsumerWarps * kMaxGroup;                    // [8][W]
#pragma unroll
    for (int e = 0; e < 2; ++e) {   // query rows 2t and 2t + 1
        const int row = 2 * t + e;
        if (row < G) {
            float *dst = red_o + (warp * kMaxGroup + row) * kRowStride;
#pragma unroll
            for (int n = 0; n < D / 16; ++n) {
                const int dim = 32 * (n >> 1) + 4 * r + 2 * (n & 1);
                *reinterpret_cast<float2 *>(dst + dim) = make_float2(o[n][e], o[n][2 + e]);
            }
        }
    }
    if (r < G && t == 0) {
        red_m[warp * kMaxGroup + r] = m_run;
        red_l[warp * kMaxGroup + r] = l_run;
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
        const float inv = (L > 0.0f) ? 1.0f / L : 0.0f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w)
            row_w[row * kConsumerWarps + w] = f[w] * inv;
        if (SPLIT)
            a.part_lse[(row0 + row) * a.n_split + split] =
                (L > 0.0f) ? (M + log2f(L)) * kLn2 : -INFINITY;
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
            const size_t prow = (row0 + row) * a.n_split + split;
            *reinterpret_cast<float4 *>(a.part_o + prow * D + c) = acc;
        } else {
            store_out4(a.out, a.out_f32, (row0 + row) * D + c, acc);
        }
    }
}

template <int D, bool SPLIT>
cudaError_t launch_t(const DecodeInt8Launch &l, const CUtensorMap &tk, const CUtensorMap &tv,
                     cudaStream_t stream)
{
    constexpr size_t kSmemBytes = I8Geom<D>::kSmemBytes;
    Args a;
    a.q = static_cast<const __nv_bfloat16 *>(l.q);
    a.k_scales = l.k_scales;
    a.v_scales = l.v_scales;
    a.out = l.out;
    a.out_f32 = l.out_f32;
    a.part_o = l.part_o;
    a.part_lse = l.part_lse;
    a.block_table = l.block_table;
    a.bt_stride = l.bt_stride;
    a.context_lens = l.context_lens;
    a.q_heads = l.q_heads;
    a.kv_heads = l.kv_heads;
    a.group = l.q_heads / l.kv_heads;
    a.page_size = l.page_size;
    a.chunk = l.chunk;
    a.n_split = l.n_split;
    a.scale_log2 = l.scale * 1.4426950408889634f;
    a.k_new = static_cast<const __nv_bfloat16 *>(l.k_new);
    a.v_new = static_cast<const __nv_bfloat16 *>(l.v_new);
    a.k_codes_w = static_cast<int8_t *>(l.k_codes_w);
    a.v_codes_w = static_cast<int8_t *>(l.v_codes_w);
    a.k_scales_w = l.k_scales_w;
    a.v_scales_w = l.v_scales_w;
    a.num_slots = l.num_slots;
    a.err = current_error_word();
    a.hnd = l.hnd ? 1 : 0;
    auto kernel = paged_decode_int8_kernel<D, SPLIT>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kSmemBytes));
    if (err != cudaSuccess)
        return err;
    dim3 grid(l.n_split, l.kv_heads, l.num_seqs);
    return launch_pdl(kernel, grid, dim3(kThreads), kSmemBytes, stream, tk, tv, a);
}

}  // namespace

cudaError_t launch_decode_int8(const DecodeInt8Launch &l, const CUtensorMap &tmap_k,
                               const CUtensorMap &tmap_v, cudaStream_t stream)
{
    if (l.num_seqs == 0)
        return cudaSuccess;
    if (l.head_dim == 64)
        return l.n_split > 1 ? launch_t<64, true>(l, tmap_k, tmap_v, stream)
                             : launch_t<64, false>(l, tmap_k, tmap_v, stream);
    return l.n_split > 1 ? launch_t<128, true>(l, tmap_k, tmap_v, stream)
                         : launch_t<128, false>(l, tmap_k, tmap_v, stream);
}

cudaError_t read_and_clear_decode_int8_errors(uint32_t *flags)
{
    uint32_t zero = 0;
    cudaError_t err = cudaMemcpyFromSymbol(flags, g_decode_int8_errors, sizeof(uint32_t));
    if (err != cudaSuccess)
        return err;
    return cudaMemcpyToSymbol(g_decode_int8_errors, &zero, sizeof(uint32_t));
}

}  // namespace kvc
