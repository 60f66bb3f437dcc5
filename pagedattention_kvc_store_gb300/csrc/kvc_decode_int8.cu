// kvc_decode_int8.cu -- paged decode attention over INT8 pages.
//
// What it computes: the attention of kvc_decode ("KV Cache Management and PagedAttention",
// "Compute attention over scattered KV") over pages that hold int8 codes with one fp32 scale
// per (position, kv head) vector (TileInfer.jl "KV cache", "INT8 cache").  As that section
// says, the cache is not dequantised: a key's scale multiplies its score, and a value's scale
// its probability before the PV product.  Codes are converted to fp16 in registers (exact:
// |code| <= 127) for the tensor cores; the scales stay outside the products.  fp16 rather than
// bf16 because four codes become two exact fp16 pairs in five integer/half operations: the
// sign bits flipped (b = code + 128), the bytes placed under the exponent 0x64 (1024 + b), and
// 1152 subtracted; the query is converted to fp16 once per piece (scaled by a power of two
// when it would overflow fp16), and the probabilities (at most 1) times the value scales enter
// the PV product as fp16.
//
// Layout: codes [num_pages * P][Hkv][D] int8 like the bf16 pools (D bytes per vector), or
// [num_pages][Hkv][P][D] (HND); scales [num_pages][Hkv][P] fp32, so the P scales of one (page,
// kv head) are one contiguous run that a single bulk copy brings in.
//
// Work partition.  The consumer warps convert every code they read, so a CTA is bound by its own
// instruction stream, not by HBM: an SM runs at the pace of its three resident CTAs, and every
// microsecond one of them spends starting up (page ids, first copies) or idle at the end of a
// ragged grid is lost.  So for each kv head the positions of all sequences, in 64-position blocks
// (sequence-major), are cut into R runs of equal cost, one per CTA (CTA = run * Hkv + kv head, R *
// Hkv = one wave of resident CTAs), a block costing 16 and each sequence start kPieceCost (a
// further piece costs its CTA about 0.9 of a block), and each CTA streams its run without a break:
// the pieces of the sequences it covers follow one another through the same ring.  The runs of all
// kv heads have the same bounds, so the CTAs that read one sequence's positions for its kv heads
// start together and stay in step (the kv heads of a position share its NHD rows; on 64 sequences
// of 512-4,096 positions 76.9 against 91.3 us for unaligned runs).  A piece that is a whole unit
// (sequence, kv head) writes the output rows; the others write a partial (rows normalised by their
// own sum, and the log-sum-exp) to slot h (S + R) + s + run of the workspace -- distinct for every
// piece, consecutive for one unit's pieces.  The merge (merge_flat_kernel) finds a unit's slots
// from the context lengths with the same cut; in batches of over kMergeScanSeqs sequences the
// unit's first piece records them (first slot, piece count) instead.  With num_splits = 1 the
// kernel instead runs one CTA per unit (no workspace, no merge).  The producer alone walks the
// runs; it hands each piece (its sequence, blocks and context) to the consumers in shared memory
// with the query rows, so all warps of a CTA take the same path whatever the context lengths.
//
// CTA: 4 consumer warps and a producer warp, three CTAs per SM.  The producer loads each
// piece's query rows into shared memory and streams 64-position stages -- per page one TMA box
// of K codes, one of V codes (128-byte swizzle at D = 128, 64-byte at D = 64) and one bulk copy
// each of the K and V scales, issued by parallel lanes -- through a 4-deep ring.  Consumer warp
// w takes positions 16 w .. 16 w + 15 of each stage:
//   S^T = K Q^T on mma.sync m16n8k16 (fp16): the warp's 16 positions are the M rows and the G
//   query heads the N columns (padded to 8).  The order in which head_dim is contracted is
//   free, so thread (r, t) takes dims (D / 4) t + 4 kk .. + 3 for k-step kk: its K codes of a
//   position are D / 4 contiguous bytes, one word per k-step, and its Q pairs are two
//   contiguous pairs;
//   O^T += V^T (P * v_scale)^T with M = 16 dims and N = 8 query heads, V^T from a transposing
//   8-bit ldmatrix (m16n16, x2: two dim tiles per load), which gives each thread the bytes of
//   positions 4t .. 4t + 3 of one dim per register, converted like K's.  The contraction over
//   the warp's 16 positions runs in that order, so contraction index k is position
//   4 ((k % 8) / 2) + 2 (k / 8) + k % 2; a thread's score rows r, r + 8 (its S^T rows, and so
//   the K rows it reads) are the positions of k = r and r + 8, and one 8x8 transpose
//   (movmatrix) per half turns its fp16 probabilities (heads 2t, 2t + 1) into the B fragment
//   of the PV product (k = 2t, 2t + 1 / 2t + 8, 2t + 9; head r).  The O^T rows a thread
//   accumulates are its own score heads 2t, 2t + 1, so the rescale needs no exchange.
// Online softmax in base 2, masked positions excluded before the exponential and their
// probabilities set to 0 by selection (a scale left in an unused slot may be NaN).  At the end
// of a piece the 4 warps combine in the buffer of the piece's last stage, which the consumers
// release only afterwards, while the producer already streams the next piece.
// Fused store (kvc_decode_int8_store): the producer of the CTA whose piece ends at a unit's
// newest position quantises that token's K/V row with the INT8 store's arithmetic and writes
// its codes and scale before the copies of that page.
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
constexpr float kLog2e = 1.4426950408889634f;

// Stage layout for head_dim D (64 or 128): K codes [64 rows][D], V codes, K scales, V scales.
// The query rows of the current piece (bf16 [G][D]) and the barriers follow the ring.
template <int D>
struct I8Geom {
    static constexpr int kCodeBytes = kStageKeys * D;        // K (or V) codes of one stage
    static constexpr int kScaleBytes = kStageKeys * 4;
    static constexpr int kOffV = kCodeBytes;
    static constexpr int kOffKs = 2 * kCodeBytes;
    static constexpr int kOffVs = kOffKs + kScaleBytes;
    static constexpr int kStageBytes = ((2 * kCodeBytes + 2 * kScaleBytes) + 1023) & ~1023;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kQBytes = kMaxGroup * D * 2;
    static constexpr int kCombineBytes =   // o rows, m, l per warp; weights per row
        kConsumerWarps * kMaxGroup * (D + 4) * 4 + 3 * kConsumerWarps * kMaxGroup * 4;
    static_assert(kCombineBytes <= kStageBytes, "combine area is one stage buffer");
    static constexpr int kBarBytes = (2 * kStages + 2) * 8;
    static constexpr int kScratchBytes = 128;   // scan sums, run start, abort flag, piece
    static constexpr size_t kSmemBytes =
        1024 + kRingBytes + kQBytes + kBarBytes + kScratchBytes;
};

// Batches of up to this many sequences: the merge finds each unit's partial slots from the
// context lengths itself, before it waits for the decode; larger ones read the slot info the
// decode wrote (a scan of every context per merge warp would grow with the square of the batch).
constexpr int kMergeScanSeqs = 256;

struct Args {
    const __nv_bfloat16 *q;
    const float *k_scales, *v_scales;
    void *out;
    int out_f32;
    float *part_o;       // [U + N][G][D] partials of the pieces that are not whole units
    float *part_lse;     // [U + N][G]
    int2 *unit_info;     // [U]: (first slot, piece count) of each non-empty unit, written
                         // for batches over kMergeScanSeqs sequences
    int runs;            // runs per kv head (the grid is runs * kv_heads CTAs)
    const int32_t *block_table;
    int bt_stride;
    const int32_t *context_lens;
    int num_seqs, q_heads, kv_heads, group, page_size;
    int per_unit;        // 1: one CTA per unit (blockIdx.x = unit), no partials
    float scale_log2;
    // kvc_decode_int8_store: sequence s's new key and value (bf16 [S][Hkv][D]), quantised and
    // written to the code and scale pools (num_slots slots) by the CTA whose piece ends at the
    // newest position, before that CTA's copies of the page; null otherwise.
    const __nv_bfloat16 *k_new, *v_new;
    int8_t *k_codes_w, *v_codes_w;
    float *k_scales_w, *v_scales_w;
    int num_slots;
    uint32_t *err;   // the caller's device error word, or null (this file's own word)
    int hnd;         // HND codes: page boxes addressed by (offset, page * kv_heads + kv head)
};

__device__ __forceinline__ uint32_t *err_word(const Args &a)
{
    return a.err ? a.err : &g_decode_int8_errors;
}

// A sequence's context as the kernel reads it: clamped to [0, bt_stride * P] (a longer one is
// flagged by CTA 0 and attends over the positions its block-table row holds, storing nothing).
__device__ __forceinline__ int clamped_ctx(const Args &a, int s, bool *over = nullptr)
{
    const int raw = a.context_lens[s];
    const int cap = a.bt_stride * a.page_size;
    if (over)
        *over = raw > cap;
    return max(0, min(raw, cap));
}

__device__ __forceinline__ int blocks_of(int ctx) { return (ctx + kStageKeys - 1) / kStageKeys; }

// A sequence's clamped context read by lane 0 of the calling warp and shared with its lanes
// (the producer's walk takes every decision once for the whole warp).
__device__ __forceinline__ int ctx_for_warp(const Args &a, int s, bool &over)
{
    int raw = 0;
    if ((threadIdx.x & 31) == 0)
        raw = a.context_lens[s];
    raw = __shfl_sync(0xffffffffu, raw, 0);
    const int cap = a.bt_stride * a.page_size;
    over = raw > cap;
    return max(0, min(raw, cap));
}

// Position of the producer's walk in its kv head's block order (sequence-major, then block).
struct Cursor {
    int s, blk;        // current sequence and its next block
    int ctx, nb;       // the sequence's (clamped) context and block count
    bool over;         // the context was past the block-table row
    long long g;       // index of the next block in the kv head's order
};

// Loads the context of cursor sequence w.s, moving past sequences with no positions; false
// when none is left (the contexts changed under the launch).
__device__ __forceinline__ bool cursor_load(Cursor &w, const Args &a)
{
    for (; w.s < a.num_seqs; ++w.s) {
        w.ctx = ctx_for_warp(a, w.s, w.over);
        w.nb = blocks_of(w.ctx);
        if (w.nb > 0)
            return true;
    }
    return false;
}

// After a piece of n blocks: the next sequence when the piece ended this one; false when the
// walk cannot go on.
__device__ __forceinline__ bool cursor_advance(Cursor &w, const Args &a, int n, long long g1)
{
    w.g += n;
    w.blk += n;
    if (w.blk == w.nb) {
        w.blk = 0;
        ++w.s;
        if (w.g < g1)
            return cursor_load(w, a);
    }
    return true;
}

// One piece as the producer hands it to the consumers (with the query rows): sequence s of the
// CTA's kv head, blocks blk0 .. blk0 + nblk - 1 of its nb, its context, and the index of its
// last block in the kv head's order; nblk = 0 ends the CTA's work.
struct PieceDesc {
    int s, blk0, nblk, ctx, nb;
    long long g_last;
};

// The cost of a piece's start against its blocks' (16 per 64-position block) when the runs are
// cut: a CTA pays about 0.9 of a block's streaming time for each further sequence its run
// holds (the combine and write-out of the piece before it, the next piece's query rows).
constexpr long long kPieceCost = 14;

// floor((x y + add) / d) for x y + add below 2^64 + 2^63 (d > 0): in 64-bit arithmetic when the
// product fits (every practical size; a 128-bit quotient is a long software routine), else in
// 128-bit.
__device__ __forceinline__ unsigned long long mul_div(unsigned long long x, unsigned long long y,
                                                      long long add, unsigned long long d)
{
    const unsigned long long lo = x * y;
    if (__umul64hi(x, y) == 0 && (add >= 0 ? lo <= ~0ull - static_cast<unsigned long long>(add)
                                           : lo >= static_cast<unsigned long long>(-add)))
        return (lo + static_cast<unsigned long long>(add)) / d;
    const __int128 num = static_cast<__int128>(static_cast<unsigned __int128>(x) * y) + add;
    return static_cast<unsigned long long>(static_cast<unsigned __int128>(num) / d);
}

// Runs are cut in cost units: block g of sequence s sits at cost 16 g + kPieceCost (s + 1)
// (strictly increasing along a kv head's block order; a kv head's T blocks over S sequences
// span C = 16 T + kPieceCost S), and run c of n holds the blocks at costs
// [floor(c C / n), floor((c + 1) C / n)).
__device__ __forceinline__ long long block_cost(long long g, int s)
{
    return 16 * g + kPieceCost * (s + 1);
}

// Start of run c of n in cost units: floor(c C / n).
__device__ __forceinline__ long long run_start(long long c, long long cost, long long n)
{
    return static_cast<long long>(mul_div(c, cost, 0, n));
}

// The run that holds cost position x: the largest c with run_start(c) <= x.
__device__ __forceinline__ long long run_of(long long x, long long cost, long long n)
{
    return static_cast<long long>(mul_div(x + 1, n, -1, cost));
}

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

// Offset of byte `col` of stage row `row` in a [64][D] code tile: 128-byte rows with the
// 128-byte swizzle (16-byte chunk c of row r at c ^ (r % 8)), or 64-byte rows with the 64-byte
// swizzle (chunk c of row r at c ^ ((r / 2) % 4)).
template <int D>
__device__ __forceinline__ uint32_t code_offset(int row, int col)
{
    const int phase = D == 128 ? (row & 7) : ((row >> 1) & 3);
    return static_cast<uint32_t>(row * D + ((((col >> 4) ^ phase)) << 4) + (col & 15));
}

template <int D>
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
    __nv_bfloat16 *qbuf = reinterpret_cast<__nv_bfloat16 *>(smem + kRingBytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kRingBytes + Geom::kQBytes);
    uint64_t *empty = full + kStages;
    uint64_t *q_full = empty + kStages;
    uint64_t *q_empty = q_full + 1;
    // [0] first sequence, [1] its first block, [2..6] scan sums, [7] g1, [9] g0
    long long *scratch = reinterpret_cast<long long *>(q_empty + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(scratch + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.group;
    const int P = a.page_size;
    const int Hkv = a.kv_heads;
    // CTA = run * Hkv + kv head: the runs of every kv head have the same bounds, so the CTAs
    // reading one sequence's pages for its kv heads start together and stay in step (the kv
    // heads of a position share its NHD rows)
    const int kvh = static_cast<int>(blockIdx.x % Hkv);
    const long long run = blockIdx.x / Hkv;
    const long long n_run_ctas = gridDim.x / Hkv;

    volatile PieceDesc *desc = reinterpret_cast<volatile PieceDesc *>(scratch + 10);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        mbar_init(q_full, 1);
        mbar_init(q_empty, kConsumerWarps);
        *abort_flag = 0;
        scratch[0] = -1;
        scratch[7] = -1;
        scratch[9] = -1;
        fence_mbar_init();
    }

    // ---- this CTA's run of blocks [g0, g1) and where it starts: sequence scratch[0], whose
    // first block has global index scratch[1] (one unit: its context scratch[1] and blocks
    // scratch[2]); g0 and g1 in scratch[9] and scratch[7].  Every decision below reads shared
    // memory, so the whole CTA takes it alike.
    long long g0 = 0, g1 = 0, total = 0;   // per kv head
    long long cost = 0;                     // the kv head's blocks and pieces in cost units
    long long n_runs = n_run_ctas;          // runs of a kv head: at most one per block
    if (a.per_unit) {
        // one unit per CTA, numbered on its own: blocks [0, nb)
        if (threadIdx.x == 0) {
            const int s0 = static_cast<int>(run);
            bool over;
            const int ctx = clamped_ctx(a, s0, &over);
            if (over && kvh == 0)
                atomicOr(err_word(a), kErrContextRange);
            scratch[0] = s0;
            scratch[1] = ctx;
            scratch[2] = blocks_of(ctx);
            scratch[3] = over;
        }
        __syncthreads();
        total = scratch[2];
        g1 = total;
        if (total == 0) {   // no positions: the rows are 0
            const size_t row0 = static_cast<size_t>(blockIdx.x) * G;
            for (int i = threadIdx.x; i < G * D; i += blockDim.x)
                store_out(a.out, a.out_f32, row0 * D + i, 0.0f);
            return;
        }
    } else {
        // block counts of all sequences, summed by a block-wide scan (every CTA computes the
        // same total, a kv head's; CTA 0 flags contexts past their block-table rows)
        const int S = a.num_seqs;
        const int per = (S + kThreads - 1) / kThreads;
        const int lo = min(S, static_cast<int>(threadIdx.x) * per);
        const int hi = min(S, lo + per);
        long long mine = 0;
        for (int s = lo; s < hi; ++s) {
            bool over;
            mine += blocks_of(clamped_ctx(a, s, &over));
            if (over && blockIdx.x == 0)
                atomicOr(err_word(a), kErrContextRange);
        }
        long long incl = mine;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off)
                incl += v;
        }
        if (lane == 31)
            scratch[2 + warp] = incl;
        __syncthreads();
        long long before = incl - mine, sum = 0;
#pragma unroll
        for (int i = 0; i < kThreads / 32; ++i) {
            const long long t = scratch[2 + i];
            if (i < warp)
                before += t;
            sum += t;
        }
        total = sum;
        n_runs = min(n_run_ctas, total);
        cost = 16 * total + kPieceCost * S;
        if (run < n_runs) {
            // the run's bounds in cost units; sequence s covers costs [kPieceCost s + 16 B_s,
            // kPieceCost (s + 1) + 16 (B_s + nb_s)) (B_s: blocks before it), which tile
            // [0, cost), so exactly one thread finds each bound below the end: the first block
            // at or past it (B_s + nb_s when it falls after s's last block)
            const long long c0 = run_start(run, cost, n_runs);
            const long long c1 = run_start(run + 1, cost, n_runs);
            long long acc = before;
            for (int s = lo; s < hi; ++s) {
                const long long nb = blocks_of(clamped_ctx(a, s));
                const long long lo_cost = kPieceCost * s + 16 * acc;
                const long long first = block_cost(acc, s);
                const long long hi_cost = first + 16 * nb;
                if (c0 >= lo_cost && c0 < hi_cost) {
                    const long long off = min(nb, max(0LL, (c0 - first + 15) / 16));
                    scratch[9] = acc + off;
                    scratch[0] = off < nb ? s : s + 1;   // empty ones are skipped by the walk
                    scratch[1] = off < nb ? acc : acc + nb;
                }
                if (c1 >= lo_cost && c1 < hi_cost)
                    scratch[7] = acc + min(nb, max(0LL, (c1 - first + 15) / 16));
                acc += nb;
            }
        }
        __syncthreads();
        g0 = scratch[9] >= 0 ? scratch[9] : total;
        g1 = scratch[7] >= 0 ? scratch[7] : total;   // the last run ends with the blocks
        if (run >= n_runs || g0 >= g1 || scratch[0] < 0 || scratch[0] >= S)
            return;   // an empty run
    }

    if (warp == kConsumerWarps) {
        // ------------------------ producer (whole warp) -------------------------------------
        if (lane == 0) {
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
        }
        const uint64_t policy = l2_policy_evict_first();
        int i = 0;   // stages issued
        int p = 0;   // pieces handed over
        bool ok = true;
        Cursor w;
        w.s = static_cast<int>(scratch[0]);
        w.g = g0;
        if (a.per_unit) {
            w.ctx = static_cast<int>(scratch[1]);
            w.nb = static_cast<int>(total);
            w.over = scratch[3] != 0;
            w.blk = 0;
        } else {
            ok = cursor_load(w, a);
            const long long off = g0 - scratch[1];
            ok = ok && off < w.nb;
            w.blk = ok ? static_cast<int>(off) : 0;
        }
        // a piece's query rows (bf16 [G][D], 16 bytes per lane and step), requested with its
        // page ids so that both round trips overlap, and stored when the piece is handed over
        constexpr int kQSteps = kMaxGroup * D / 8 / 32;
        uint4 q_rows[kQSteps];
        auto load_q = [&](int s) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                a.q + (static_cast<size_t>(s) * a.q_heads + static_cast<size_t>(kvh) * G) * D);
#pragma unroll
            for (int k = 0; k < kQSteps; ++k)
                if (lane + 32 * k < G * D / 8)
                    q_rows[k] = src[lane + 32 * k];
        };
        // hands piece p (nblk = 0: the end) over with its query rows, once the consumers have
        // taken piece p - 1's
        auto hand_over = [&](int s, int blk0, int nblk, int ctx, int nb) -> bool {
            if (p > 0 && !__all_sync(0xffffffffu, mbar_wait(q_empty, (p - 1) & 1)))
                return false;
            if (nblk > 0) {
                uint4 *dst = reinterpret_cast<uint4 *>(qbuf);
#pragma unroll
                for (int k = 0; k < kQSteps; ++k)
                    if (lane + 32 * k < G * D / 8)
                        dst[lane + 32 * k] = q_rows[k];
            }
            if (lane == 0) {
                desc->s = s;
                desc->blk0 = blk0;
                desc->nblk = nblk;
                desc->ctx = ctx;
                desc->nb = nb;
                desc->g_last = w.g - blk0 + nb - 1;
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(q_full);
            ++p;
            return true;
        };
        // per-lane constants of the copies: lane 4 j + op issues page j's K codes (op 0), V
        // codes (1), K scales (2) or V scales (3); page sizes are powers of two
        const int shP = __ffs(P) - 1;
        const int j = lane >> 2;
        const int op = lane & 3;
        const uint32_t dst_off = op == 0   ? j * P * D
                                 : op == 1 ? kOffV + j * P * D
                                 : op == 2 ? kOffKs + j * P * 4
                                           : kOffVs + j * P * 4;
        const float *scale_base = op == 2 ? a.k_scales : a.v_scales;
        const int c1 = a.hnd ? 0 : kvh;
        while (ok && w.g < g1) {
            const int blk0 = w.blk;
            const int nblk = static_cast<int>(min(static_cast<long long>(w.nb - blk0), g1 - w.g));
            const int s = w.s, ctx = w.ctx;
            if (nblk <= 0) {
                ok = false;
                break;
            }
            load_q(s);
            const int32_t *bt_row = a.block_table + static_cast<size_t>(s) * a.bt_stride;
            const int unit_pages = (ctx + P - 1) >> shP;
            // page ids in windows of 32 (one per lane), the next window requested one window
            // ahead; a stage's pages never straddle two windows (64 / P divides 32)
            int cached_base = blk0 << (6 - shP);
            int cached_page = cached_base + lane < unit_pages ? bt_row[cached_base + lane] : 0;
            int next_page =
                cached_base + 32 + lane < unit_pages ? bt_row[cached_base + 32 + lane] : 0;
            // this piece writes the new token when it ends at the unit's newest position:
            // before the last stage's copies read that page's codes and scales
            const bool writes_new = a.k_new != nullptr && !w.over && blk0 + nblk == w.nb;
            uint32_t k_row_new[E / 2] = {}, v_row_new[E / 2] = {};
            int new_page = 0;
            if (writes_new) {
                const size_t src = ((static_cast<size_t>(s) * Hkv + kvh) * 32 + lane) * (E / 2);
                const uint32_t *kn = reinterpret_cast<const uint32_t *>(a.k_new) + src;
                const uint32_t *vn = reinterpret_cast<const uint32_t *>(a.v_new) + src;
#pragma unroll
                for (int e = 0; e < E / 2; ++e) {
                    k_row_new[e] = __ldg(kn + e);
                    v_row_new[e] = __ldg(vn + e);
                }
                new_page = bt_row[(ctx - 1) >> shP];
            }
            for (int b = 0; b < nblk; ++b) {
                const int st = i % kStages;
                if (i >= kStages &&
                    !__all_sync(0xffffffffu, mbar_wait(&empty[st], ((i / kStages) - 1) & 1))) {
                    ok = false;
                    break;
                }
                const int blk = blk0 + b;
                const int keys = min(kStageKeys, ctx - blk * kStageKeys);
                const int np = (keys + P - 1) >> shP;
                if (lane == 0)
                    mbar_arrive_expect_tx(&full[st],
                                          static_cast<uint32_t>((np << shP) * (2 * D + 2 * 4)));
                __syncwarp();
                uint8_t *stage = smem + st * kStageBytes;
                const int lp0 = blk << (6 - shP);
                if (lp0 >= cached_base + 32) {
                    cached_base += 32;
                    cached_page = next_page;
                    next_page = cached_base + 32 + lane < unit_pages
                                    ? bt_row[cached_base + 32 + lane]
                                    : 0;
                }
                const int page = __shfl_sync(0xffffffffu, cached_page, (lp0 - cached_base + j) & 31);
                if (writes_new && b + 1 == nblk) {
                    const int off_new = (ctx - 1) % P;
                    const long long slot = static_cast<long long>(new_page) * P + off_new;
                    if (new_page >= 0 && slot < a.num_slots) {
                        const size_t sidx =
                            (static_cast<size_t>(new_page) * Hkv + kvh) * P + off_new;
                        const size_t row =
                            (a.hnd ? sidx : static_cast<size_t>(slot) * Hkv + kvh) * D;
                        quantise_store_row<E>(k_row_new, a.k_codes_w + row, a.k_scales_w + sidx,
                                              lane);
                        quantise_store_row<E>(v_row_new, a.v_codes_w + row, a.v_scales_w + sidx,
                                              lane);
                    } else if (lane == 0) {
                        atomicOr(err_word(a), kErrSlotRange);   // skipped, as in the store
                    }
                    // the stores (generic proxy) before the copies (async proxy) that read them
                    fence_proxy_async_global();
                    __syncwarp();
                    fence_proxy_async_global();
                }
                if (j < np) {
                    const int pk = page * Hkv + kvh;   // (page, kv head): scales, HND boxes
                    if (op < 2)
                        tma_load_3d(stage + dst_off, op == 0 ? &tmap_k : &tmap_v, 0, c1,
                                    a.hnd ? pk : page << shP, &full[st], policy);
                    else
                        bulk_load(stage + dst_off, scale_base + (static_cast<size_t>(pk) << shP),
                                  P * 4, &full[st]);
                }
                ++i;
                // the piece goes to the consumers once its first stage is on its way
                if (b == 0 && !hand_over(s, blk0, nblk, ctx, w.nb)) {
                    ok = false;
                    break;
                }
            }
            if (!ok)
                break;
            ok = cursor_advance(w, a, nblk, g1);
        }
        if (ok)
            ok = hand_over(0, 0, 0, 0, 0);   // the end
        if (!ok && lane == 0) {
            atomicOr(err_word(a), kErrDecodeEmptyWait);
            for (int b = max(0, i - kStages); b < i; ++b)
                if (!mbar_wait(&full[b % kStages], (b / kStages) & 1))
                    atomicOr(err_word(a), kErrDrainWait);
        }
        return;
    }

    // --------------------------------- consumers -----------------------------------------
    const int r = lane >> 2;   // fragment group: contraction rows r, r + 8; query head r
    const int t = lane & 3;
    const int wrow = warp * kKeysPerWarp;   // first stage row of this warp
    // The PV product's contraction index k (0..15) runs over this warp's positions in the
    // order in which a transposing ldmatrix hands V over: thread (g, t) gets, per dim, the
    // bytes of positions 4t .. 4t + 3, whose pairs are its A fragment's k = 2t, 2t + 1 and
    // 2t + 8, 2t + 9.  So k is position pk(k) = 4 ((k % 8) / 2) + 2 (k / 8) + k % 2, and the
    // S^T rows r, r + 8 of this thread (k = r, r + 8, the movmatrix hands them over as k) are
    // positions pos0 = pk(r) and pos1 = pos0 + 2.
    const int pos0 = 4 * (r >> 1) + (r & 1);
    const int pos1 = pos0 + 2;
    // Stage-independent offsets.  K: the 16-byte chunks of this thread's D / 4 bytes in rows
    // wrow + pos0 and wrow + pos1.  V: lane l's row address of each ldmatrix.x2 (matrices of 16
    // positions x 16 dims: row l % 16 of matrix 2 m + l / 16, 16-byte chunk 2 m + l / 16).
    constexpr int kKChunks = D / 64;   // 16-byte chunks of this thread's K bytes per row
    constexpr int kVPairs = D / 32;    // ldmatrix.x2 loads per stage (two 16-dim tiles each)
    uint32_t k_off[2][kKChunks];
#pragma unroll
    for (int h = 0; h < kKChunks; ++h) {
        k_off[0][h] = code_offset<D>(wrow + pos0, (D / 4) * t + 16 * h);
        k_off[1][h] = code_offset<D>(wrow + pos1, (D / 4) * t + 16 * h);
    }
    uint32_t v_ldm[kVPairs];
#pragma unroll
    for (int m = 0; m < kVPairs; ++m)
        v_ldm[m] = kOffV + code_offset<D>(wrow + (lane & 15), 16 * (2 * m + (lane >> 4)));
    const uint32_t smem32 = smem_addr(smem);
    constexpr int kRowStride = D + 4;
    bool ok = true;
    int i = 0;   // stages consumed
    int p = 0;   // pieces begun

    while (true) {
        // the next piece and its query rows.  Q^T pairs (the B fragment of S^T = K Q^T, column
        // r = query head r, rows >= G padding) in the contraction order (k-step kk uses dims
        // (D / 4) t + 4 kk + {0, 1} and {2, 3}), as fp16.  A power of two q_pow brings the
        // largest |q| of the group below 2^14 when it is above, and is folded back into the
        // score scale (exact either way).
        const bool q_ok = __all_sync(0xffffffffu, mbar_wait(q_full, p & 1));
        const int s = desc->s, blk0 = desc->blk0, nblk = desc->nblk;
        const int ctx = desc->ctx, nb = desc->nb;
        const long long g_last = desc->g_last;
        uint32_t qa[D / 16][2];
        float sl2 = a.scale_log2;
        {
            float qv[D / 4];
            const uint4 *qrow = reinterpret_cast<const uint4 *>(qbuf + r * D + (D / 4) * t);
#pragma unroll
            for (int k = 0; k < D / 32; ++k) {
                uint4 w4 = make_uint4(0u, 0u, 0u, 0u);
                if (r < G && q_ok)
                    w4 = qrow[k];
                const uint32_t wd[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    qv[8 * k + 2 * e] = __uint_as_float(wd[e] << 16);
                    qv[8 * k + 2 * e + 1] = __uint_as_float(wd[e] & 0xFFFF0000u);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(q_empty);
            if (!q_ok)
                *abort_flag = 1;
            // one decision for the 4 warps: stop on a wait that gave up, or at the end
            named_barrier(1, kConsumerWarps * 32);
            if (*abort_flag || nblk <= 0)
                break;
            float qmax = 0.0f;
#pragma unroll
            for (int k = 0; k < D / 4; ++k)
                qmax = fmaxf(qmax, fabsf(qv[k]));
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
        const bool whole = blk0 == 0 && nblk == nb;
        const int unit = s * Hkv + kvh;
        const size_t row0 = static_cast<size_t>(s) * a.q_heads + static_cast<size_t>(kvh) * G;
        // O^T accumulators: tile n holds dims 16 n .. 16 n + 15 x query heads, this thread
        // heads 2t, 2t + 1 of dims 16 n + r (c0, c1) and 16 n + r + 8 (c2, c3)
        float o[D / 16][4];
#pragma unroll
        for (int n = 0; n < D / 16; ++n)
            o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
        // running max and row sum of query heads 2t and 2t + 1 (the heads of this thread's
        // scores and of its O^T accumulators)
        float m_run[2] = {-INFINITY, -INFINITY};
        float l_run[2] = {0.0f, 0.0f};
        int last_st = -1;

        for (int b = 0; ok && b < nblk; ++b) {
            const int st = i % kStages;
            if (!__all_sync(0xffffffffu, mbar_wait(&full[st], (i / kStages) & 1))) {
                ok = false;
                break;
            }
            const uint8_t *stage = smem + st * kStageBytes;
            const float *ks = reinterpret_cast<const float *>(stage + kOffKs) + wrow;
            const float *vs = reinterpret_cast<const float *>(stage + kOffVs) + wrow;
            const int n_valid = ctx - ((blk0 + b) * kStageKeys + wrow);
            if (n_valid > 0) {
                // S^T = K Q^T: A rows r and r + 8 are positions pos0 and pos1 of this warp
                // (a0, a2 from one word of position pos0, a1, a3 from pos1), two chains
                float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int h = 0; h < kKChunks; ++h) {
                    const uint4 c0 = *reinterpret_cast<const uint4 *>(stage + k_off[0][h]);
                    const uint4 c1 = *reinterpret_cast<const uint4 *>(stage + k_off[1][h]);
                    const uint32_t w0[4] = {c0.x, c0.y, c0.z, c0.w};
                    const uint32_t w1[4] = {c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t a0, a1, a2, a3;
                        codes_word_f16x2(w0[j], a0, a2);
                        codes_word_f16x2(w1[j], a1, a3);
                        mma_f16_16816(sc[j & 1], a0, a1, a2, a3, qa[4 * h + j][0],
                                      qa[4 * h + j][1]);
                    }
                }
                // x[0], x[1]: position pos0, heads 2t, 2t + 1; x[2], x[3]: position pos1;
                // key-scaled
                const bool v0 = pos0 < n_valid, v1 = pos1 < n_valid;
                const float ks0 = v0 ? ks[pos0] * sl2 : 0.0f, ks1 = v1 ? ks[pos1] * sl2 : 0.0f;
                float x[4];
                x[0] = v0 ? (sc[0][0] + sc[1][0]) * ks0 : -INFINITY;
                x[1] = v0 ? (sc[0][1] + sc[1][1]) * ks0 : -INFINITY;
                x[2] = v1 ? (sc[0][2] + sc[1][2]) * ks1 : -INFINITY;
                x[3] = v1 ? (sc[0][3] + sc[1][3]) * ks1 : -INFINITY;
                float mb0 = fmaxf(x[0], x[2]), mb1 = fmaxf(x[1], x[3]);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mb0 = fmaxf(mb0, __shfl_xor_sync(0xffffffffu, mb0, off));
                    mb1 = fmaxf(mb1, __shfl_xor_sync(0xffffffffu, mb1, off));
                }
                const float mn0 = fmaxf(m_run[0], mb0), mn1 = fmaxf(m_run[1], mb1);
                if (__any_sync(0xffffffffu, mn0 > m_run[0] || mn1 > m_run[1])) {
                    const float a0 = (m_run[0] == -INFINITY) ? 0.0f : fast_exp2(m_run[0] - mn0);
                    const float a1 = (m_run[1] == -INFINITY) ? 0.0f : fast_exp2(m_run[1] - mn1);
#pragma unroll
                    for (int n = 0; n < D / 16; ++n) {
                        o[n][0] *= a0;
                        o[n][1] *= a1;
                        o[n][2] *= a0;
                        o[n][3] *= a1;
                    }
                    l_run[0] *= a0;
                    l_run[1] *= a1;
                    m_run[0] = mn0;
                    m_run[1] = mn1;
                }
                const float mu0 = (m_run[0] == -INFINITY) ? 0.0f : m_run[0];
                const float mu1 = (m_run[1] == -INFINITY) ? 0.0f : m_run[1];
                const float p0 = fast_exp2(x[0] - mu0), p1 = fast_exp2(x[1] - mu1);
                const float p2 = fast_exp2(x[2] - mu0), p3 = fast_exp2(x[3] - mu1);
                l_run[0] += p0 + p2;
                l_run[1] += p1 + p3;
                const float vs0 = v0 ? vs[pos0] : 0.0f, vs1 = v1 ? vs[pos1] : 0.0f;
                // P' = P * v_scale as fp16 pairs (k = r or r + 8; heads 2t, 2t + 1), turned by
                // an 8x8 transpose into the B fragment of the PV product (k = 2t, 2t + 1 or
                // 2t + 8, 2t + 9; head r)
                const uint32_t pa0 =
                    movmatrix_trans(pack_f16x2(v0 ? p0 * vs0 : 0.0f, v0 ? p1 * vs0 : 0.0f));
                const uint32_t pa2 =
                    movmatrix_trans(pack_f16x2(v1 ? p2 * vs1 : 0.0f, v1 ? p3 * vs1 : 0.0f));
                // O^T += V^T P'^T, A = V^T (16 dims x 16 positions): each transposed load gives
                // two dim tiles; the bytes of positions 4t .. 4t + 3 of dim 16 n + r (and
                // + 8) become a0, a2 (a1, a3) exactly as K's do
                const uint32_t vbase = smem32 + st * kStageBytes;
#pragma unroll
                for (int m = 0; m < kVPairs; ++m) {
                    uint32_t e0, e1, e2, e3;
                    ldsm_x2_trans_b8(vbase + v_ldm[m], e0, e1, e2, e3);
                    uint32_t a0, a1, a2, a3;
                    codes_word_f16x2(e0, a0, a2);
                    codes_word_f16x2(e1, a1, a3);
                    mma_f16_16816(o[2 * m], a0, a1, a2, a3, pa0, pa2);
                    codes_word_f16x2(e2, a0, a2);
                    codes_word_f16x2(e3, a1, a3);
                    mma_f16_16816(o[2 * m + 1], a0, a1, a2, a3, pa0, pa2);
                }
            }
            last_st = st;
            ++i;
            if (b + 1 < nblk) {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&empty[st]);
            }
        }

        // --------------- combine the 4 warps' results in the last stage's buffer ----------
        // Each warp leaves its unnormalised o rows (D + 4 floats apart: 16-byte aligned rows),
        // running max and row sum; one thread per query head folds them into weights
        // 2^(m_w - M) / L, and the rows are written as float4 (bf16x4) pieces: the output
        // when the piece is the whole unit, else its partial slot.
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], off);
            l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], off);
        }
        const int cst = last_st >= 0 ? last_st : 0;
        float *red_o = reinterpret_cast<float *>(smem + cst * kStageBytes);   // [W][8][D + 4]
        float *red_m = red_o + kConsumerWarps * kMaxGroup * kRowStride;       // [W][8]
        float *red_l = red_m + kConsumerWarps * kMaxGroup;                    // [W][8]
        float *row_w = red_l + kConsumerWarps * kMaxGroup;                    // [8][W]
        named_barrier(1, kConsumerWarps * 32);   // every warp is done reading that stage
#pragma unroll
        for (int e = 0; e < 2; ++e) {   // query heads 2t and 2t + 1
            const int row = 2 * t + e;
            if (row < G) {
                float *dst = red_o + (warp * kMaxGroup + row) * kRowStride;
#pragma unroll
                for (int n = 0; n < D / 16; ++n) {
                    dst[16 * n + r] = o[n][e];
                    dst[16 * n + r + 8] = o[n][2 + e];
                }
                if (r == 0) {
                    red_m[warp * kMaxGroup + row] = m_run[e];
                    red_l[warp * kMaxGroup + row] = l_run[e];
                }
            }
        }
        // partial slots: kv head h owns [h (S + R), (h + 1) (S + R)), piece (s, run) is
        // slot s + run there -- distinct for every piece, consecutive for one unit's pieces
        const int slot = kvh * (a.num_seqs + static_cast<int>(n_run_ctas)) + s + static_cast<int>(run);
        named_barrier(1, kConsumerWarps * 32);
        if (threadIdx.x < G) {
            const int row = threadIdx.x;
            float M = -INFINITY;
#pragma unroll
            for (int k = 0; k < kConsumerWarps; ++k)
                M = fmaxf(M, red_m[k * kMaxGroup + row]);
            float f[kConsumerWarps];
            float L = 0.0f;
#pragma unroll
            for (int k = 0; k < kConsumerWarps; ++k) {
                const float mw = red_m[k * kMaxGroup + row];
                f[k] = (mw == -INFINITY) ? 0.0f : fast_exp2(mw - M);
                L += f[k] * red_l[k * kMaxGroup + row];
            }
            const float inv = (L > 0.0f) ? 1.0f / L : 0.0f;
#pragma unroll
            for (int k = 0; k < kConsumerWarps; ++k)
                row_w[row * kConsumerWarps + k] = f[k] * inv;
            if (!whole)
                a.part_lse[static_cast<size_t>(slot) * G + row] =
                    (L > 0.0f) ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
        named_barrier(1, kConsumerWarps * 32);
        constexpr int kVec = D / 4;
        for (int idx = threadIdx.x; idx < G * kVec; idx += kConsumerWarps * 32) {
            const int row = idx / kVec;
            const int col = (idx - row * kVec) * 4;
            float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
            for (int k = 0; k < kConsumerWarps; ++k) {
                const float wt = row_w[row * kConsumerWarps + k];
                const float4 v = *reinterpret_cast<const float4 *>(
                    red_o + (k * kMaxGroup + row) * kRowStride + col);
                acc.x = fmaf(wt, v.x, acc.x);
                acc.y = fmaf(wt, v.y, acc.y);
                acc.z = fmaf(wt, v.z, acc.z);
                acc.w = fmaf(wt, v.w, acc.w);
            }
            if (whole)
                store_out4(a.out, a.out_f32, (row0 + row) * D + col, acc);
            else
                *reinterpret_cast<float4 *>(a.part_o + (static_cast<size_t>(slot) * G + row) * D +
                                            col) = acc;
        }
        // the unit's first piece: where its pieces are and how many (the CTA runs holding
        // its first and last blocks), for the merge of a batch too large to find them itself
        if (threadIdx.x == 0 && blk0 == 0 && !a.per_unit && a.num_seqs > kMergeScanSeqs) {
            const long long last = run_of(block_cost(g_last, s), cost, n_runs);
            a.unit_info[unit] = make_int2(slot, static_cast<int>(last - run + 1));
        }
        if (!ok)
            *abort_flag = 1;
        named_barrier(1, kConsumerWarps * 32);   // the buffer is read: the stage goes back
        if (ok && lane == 0 && last_st >= 0)
            mbar_arrive(&empty[cst]);
        if (*abort_flag)
            break;
        ++p;
    }
    if (!ok)
        atomicOr(err_word(a), kErrDecodeFullWait);
}

// One warp per output row (sequence s, query head h of unit u = (s, h / G)): the log-sum-exp
// combination of the unit's partial slots first .. first + count - 1, rows normalised by their
// own sums.  Rows of a unit whose only piece wrote them are left alone; rows of a sequence
// with no positions are 0.
template <int D>
__global__ void __launch_bounds__(128) merge_flat_kernel(const Args a)
{
    constexpr int V = D / 32;
    constexpr int kPre = 4;   // pieces whose rows are requested together with the lse values
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_rows = a.num_seqs * a.q_heads;
    const int row = blockIdx.x * 4 + warp;
    const int s = min(row, n_rows - 1) / a.q_heads;
    const int h = min(row, n_rows - 1) - s * a.q_heads;
    const int G = a.group;
    const int kvh = h / G;
    const int unit = s * a.kv_heads + kvh;
    const int g = h - kvh * G;
    // Launched as a dependent of the decode, the merge's CTAs reach the wait below while the
    // decode's last CTAs still run: a small batch's slot ranges (from the context lengths,
    // which the decode does not write) are found before it.
    const int ctx = clamped_ctx(a, s);
    int first = 0, count = 0;   // the unit's partial slots
    const bool scan = a.num_seqs <= kMergeScanSeqs;
    if (scan) {
        // blocks before sequence s and all of them (the same for every kv head), summed by the
        // warp; then the runs holding s's first and last blocks, cut as the decode cut them
        long long total = 0, before = 0;
        for (int t = lane; t < a.num_seqs; t += 32) {
            const long long nb = blocks_of(clamped_ctx(a, t));
            total += nb;
            before += t < s ? nb : 0;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            total += __shfl_xor_sync(0xffffffffu, total, off);
            before += __shfl_xor_sync(0xffffffffu, before, off);
        }
        const int nb = blocks_of(ctx);
        if (nb > 0) {
            const long long R = a.runs;
            const long long n_runs = min(R, total);
            const long long cost = 16 * total + kPieceCost * a.num_seqs;
            const long long r0 = run_of(block_cost(before, s), cost, n_runs);
            const long long r1 = run_of(block_cost(before + nb - 1, s), cost, n_runs);
            first = static_cast<int>(kvh * (a.num_seqs + R) + s + r0);
            count = static_cast<int>(r1 - r0 + 1);
        }
    }
    pdl_wait();
    pdl_trigger();
    if (row >= n_rows)
        return;
    if (!scan && ctx > 0) {
        // a unit with no positions has no pieces, and its slot info is never written
        const int2 info = a.unit_info[unit];
        first = info.x;
        count = info.y;
    }
    float acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v)
        acc[v] = 0.0f;
    float sum = 0.0f;
    if (ctx > 0) {
        if (count == 1)
            return;   // the unit's only piece wrote the rows
        const float *lse = a.part_lse + static_cast<size_t>(first) * G + g;
        const float *po = a.part_o + (static_cast<size_t>(first) * G + g) * D + lane * V;
        // one round trip after the wait: every piece's lse (lane j holds piece j, j + 32,
        // ...) and the first kPre pieces' rows
        float pre[kPre][V];
#pragma unroll
        for (int j = 0; j < kPre; ++j)
            if (j < count) {
#pragma unroll
                for (int v = 0; v < V; ++v)
                    pre[j][v] = __ldcg(po + static_cast<size_t>(j) * G * D + v);
            }
        float M = -INFINITY;
        const float mine = lane < count ? __ldcg(lse + static_cast<size_t>(lane) * G) : -INFINITY;
        M = mine;
        for (int j = lane + 32; j < count; j += 32)
            M = fmaxf(M, __ldcg(lse + static_cast<size_t>(j) * G));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        if (M != -INFINITY) {
#pragma unroll
            for (int j = 0; j < kPre; ++j) {
                if (j < count) {
                    const float wj = fast_exp2((__shfl_sync(0xffffffffu, mine, j) - M) * kLog2e);
                    sum += wj;
#pragma unroll
                    for (int v = 0; v < V; ++v)
                        acc[v] = fmaf(wj, pre[j][v], acc[v]);
                }
            }
            for (int j = kPre; j < count; ++j) {
                const float lj = j < 32 ? __shfl_sync(0xffffffffu, mine, j)
                                        : __ldcg(lse + static_cast<size_t>(j) * G);
                const float wj = fast_exp2((lj - M) * kLog2e);
                sum += wj;
                const float *src = po + static_cast<size_t>(j) * G * D;
#pragma unroll
                for (int v = 0; v < V; ++v)
                    acc[v] = fmaf(wj, __ldcg(src + v), acc[v]);
            }
        }
    }
    const float inv = sum > 0.0f ? 1.0f / sum : 0.0f;
    const size_t o = static_cast<size_t>(row) * D + lane * V;
    if constexpr (V == 4) {
        store_out4(a.out, a.out_f32, o,
                   make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv));
    } else {
#pragma unroll
        for (int v = 0; v < V; ++v)
            store_out(a.out, a.out_f32, o + v, acc[v] * inv);
    }
}

template <int D>
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
    a.unit_info = static_cast<int2 *>(l.unit_info);
    a.runs = l.per_unit ? 0 : l.n_ctas / l.kv_heads;
    a.block_table = l.block_table;
    a.bt_stride = l.bt_stride;
    a.context_lens = l.context_lens;
    a.num_seqs = l.num_seqs;
    a.q_heads = l.q_heads;
    a.kv_heads = l.kv_heads;
    a.group = l.q_heads / l.kv_heads;
    a.page_size = l.page_size;
    a.per_unit = l.per_unit ? 1 : 0;
    a.scale_log2 = l.scale * kLog2e;
    a.k_new = static_cast<const __nv_bfloat16 *>(l.k_new);
    a.v_new = static_cast<const __nv_bfloat16 *>(l.v_new);
    a.k_codes_w = static_cast<int8_t *>(l.k_codes_w);
    a.v_codes_w = static_cast<int8_t *>(l.v_codes_w);
    a.k_scales_w = l.k_scales_w;
    a.v_scales_w = l.v_scales_w;
    a.num_slots = l.num_slots;
    a.err = current_error_word();
    a.hnd = l.hnd ? 1 : 0;
    auto kernel = paged_decode_int8_kernel<D>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kSmemBytes));
    if (err != cudaSuccess)
        return err;
    const unsigned grid = l.per_unit ? static_cast<unsigned>(l.num_seqs * l.kv_heads)
                                     : static_cast<unsigned>(l.n_ctas);
    err = launch_pdl(kernel, dim3(grid), dim3(kThreads), kSmemBytes, stream, tk, tv, a);
    if (err != cudaSuccess || l.per_unit)
        return err;
    const int rows = l.num_seqs * l.q_heads;
    return launch_pdl(merge_flat_kernel<D>, dim3((rows + 3) / 4), dim3(128), 0, stream, a);
}

}  // namespace

cudaError_t launch_decode_int8(const DecodeInt8Launch &l, const CUtensorMap &tmap_k,
                               const CUtensorMap &tmap_v, cudaStream_t stream)
{
    if (l.num_seqs == 0)
        return cudaSuccess;
    if (l.head_dim == 64)
        return launch_t<64>(l, tmap_k, tmap_v, stream);
    return launch_t<128>(l, tmap_k, tmap_v, stream);
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
