// kvc_store.cu -- slot mapping and the paged KV store.
//
// Slot mapping: TileInfer.jl "KV cache", "Pages and block tables" (a token's slot is its
// page from the block table times the page size, plus its offset in the page).
// Store: same section (the new keys and values are written at their slots) and "KV Cache
// Management and PagedAttention", "Grow the allocation as generation proceeds".
//
// Both are HBM-bound copies.  The store moves each token's (kv_heads * head_dim) bf16 row
// -- contiguous in the NHD pool -- with 16-byte vector loads and stores, one thread per
// 16-byte chunk, grid-stride over a grid sized in multiples of the SM count.
#include "kvc_device.cuh"
#include "kvc_launch.h"

namespace kvc {

namespace {

__device__ uint32_t g_store_errors;

// One thread per new token of a decode batch (one new token per sequence).
__global__ void slot_mapping_decode_kernel(int32_t *__restrict__ slots,
                                           const int32_t *__restrict__ block_table,
                                           int bt_stride,
                                           const int32_t *__restrict__ context_lens,
                                           int num_seqs, int page_size, uint32_t *word)
{
    pdl_wait();
    pdl_trigger();
    uint32_t *err = word ? word : &g_store_errors;
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= num_seqs)
        return;
    const int position = context_lens[s] - 1;
    int slot = -1;
    if (position >= bt_stride * page_size) {
        atomicOr(err, kErrContextRange);
    } else if (position >= 0) {
        const int page = block_table[static_cast<size_t>(s) * bt_stride + position / page_size];
        slot = page * page_size + position % page_size;
    }
    slots[s] = slot;
}

// One block per sequence, threads over its new tokens.
__global__ void slot_mapping_ragged_kernel(int32_t *__restrict__ slots,
                                           const int32_t *__restrict__ block_table,
                                           int bt_stride,
                                           const int32_t *__restrict__ context_lens,
                                           const int32_t *__restrict__ q_indptr,
                                           int page_size, uint32_t *word)
{
    pdl_wait();
    pdl_trigger();
    uint32_t *err = word ? word : &g_store_errors;
    const int s = blockIdx.x;
    const int first = q_indptr[s];
    const int q_len = q_indptr[s + 1] - first;
    const int ctx = context_lens[s];
    const int32_t *row = block_table + static_cast<size_t>(s) * bt_stride;
    for (int i = threadIdx.x; i < q_len; i += blockDim.x) {
        const int position = ctx - q_len + i;
        int slot = -1;
        if (position >= bt_stride * page_size)
            atomicOr(err, kErrContextRange);
        else if (position >= 0)
            slot = row[position / page_size] * page_size + position % page_size;
        slots[first + i] = slot;
    }
}

// chunks = kv_heads * head_dim * 2 / 16 per token row.
// HND pools (hnd = true): the chunk's kv head h = c / row_chunks is its own block per page,
// [page][h][offset][head_dim], so the destination is ((page * Hkv + h) * P + offset) rows of
// head_dim values.
__global__ void __launch_bounds__(256) store_kernel(uint4 *__restrict__ k_pool,
                                                    uint4 *__restrict__ v_pool,
                                                    const uint4 *__restrict__ k_new,
                                                    const uint4 *__restrict__ v_new,
                                                    const int32_t *__restrict__ slots,
                                                    int num_tokens, int chunks, int num_slots,
                                                    bool hnd, int kv_heads, int page_size,
                                                    uint32_t *word)
{
    pdl_wait();
    pdl_trigger();
    uint32_t *err = word ? word : &g_store_errors;
    const int row_chunks = chunks / kv_heads;   // 16-byte chunks of one head_dim vector
    const size_t total = static_cast<size_t>(num_tokens) * chunks;
    const size_t step = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += step) {
        const int t = static_cast<int>(i / chunks);
        const int c = static_cast<int>(i - static_cast<size_t>(t) * chunks);
        const int slot = __ldg(slots + t);
        if (slot < 0)
            continue;
        if (slot >= num_slots) {   // past the pool: skip the token, flag the call
            if (c == 0)
                atomicOr(err, kErrSlotRange);
            continue;
        }
        size_t dst = static_cast<size_t>(slot) * chunks + c;
        if (hnd) {
            const int page = slot / page_size;
            const int h = c / row_chunks;
            const size_t row =
                (static_cast<size_t>(page) * kv_heads + h) * page_size + (slot - page * page_size);
            dst = row * row_chunks + (c - h * row_chunks);
        }
        const uint4 kv = load_streaming(k_new + i);
        const uint4 vv = load_streaming(v_new + i);
        k_pool[dst] = kv;
        v_pool[dst] = vv;
    }
}

// Fused store + append, first part: the chunk's tokens in the page of its first token when
// that page also holds cached positions (positions base .. min(ctx, (base / P + 1) P) - 1 with
// base = ctx - q_len not a multiple of P), stored at their slots; the fused append reads that
// page from the pool and writes every later page of the chunk itself.  With `whole`, every
// token of the chunk (positions base .. ctx - 1, each at the page its block table lists) is
// stored and the plain append follows.  One CTA per sequence (grid-stride), one thread per
// 16-byte chunk of a token row; addressing as store_kernel.
//
// A context longer than the block-table row (ctx > bt_stride * P) is the caller's error; the
// pools then end as slot mapping + store leave them: every chunk token whose position the row
// covers is stored at its own slot (the whole chunk is handled here, and the fused append
// writes nothing for that sequence), the others are skipped, and kErrContextRange is set.
__global__ void __launch_bounds__(256) store_boundary_kernel(
    uint4 *__restrict__ k_pool, uint4 *__restrict__ v_pool, const uint4 *__restrict__ k_new,
    const uint4 *__restrict__ v_new, const int32_t *__restrict__ block_table, int bt_stride,
    const int32_t *__restrict__ q_indptr, const int32_t *__restrict__ context_lens, int num_seqs,
    int chunks, int kv_heads, int page_size, int num_slots, bool hnd, bool whole, uint32_t *word)
{
    pdl_wait();
    pdl_trigger();
    uint32_t *err = word ? word : &g_store_errors;
    const int row_chunks = chunks / kv_heads;
    const int capacity = bt_stride * page_size;   // positions a block-table row covers
    for (int s = blockIdx.x; s < num_seqs; s += gridDim.x) {
        const int tok0 = __ldg(q_indptr + s);
        const int q_len = __ldg(q_indptr + s + 1) - tok0;
        const int ctx = __ldg(context_lens + s);
        const int base = ctx - q_len;
        const bool over = ctx > capacity;
        const bool all = whole || over;   // every token of the chunk is stored here
        if (over && threadIdx.x == 0)
            atomicOr(err, kErrContextRange);
        if (q_len <= 0 || (!all && (base <= 0 || base % page_size == 0)))
            continue;
        const int n_tok = all ? q_len : min(ctx, (base / page_size + 1) * page_size) - base;
        const int32_t *bt_row = block_table + static_cast<size_t>(s) * bt_stride;
        const int page0 = all ? 0 : __ldg(bt_row + base / page_size);
        for (int i = threadIdx.x; i < n_tok * chunks; i += blockDim.x) {
            const int t = i / chunks;
            const int c = i - t * chunks;
            const int pos = base + t;
            if (pos < 0 || pos >= capacity)
                continue;   // no slot: before position 0, or past the block-table row
            const int page = all ? __ldg(bt_row + pos / page_size) : page0;
            const long long slot = static_cast<long long>(page) * page_size + pos % page_size;
            if (slot < 0 || slot >= num_slots) {   // a page outside the pool: skip, flag
                if (c == 0)
                    atomicOr(err, kErrSlotRange);
                continue;
            }
            size_t dst = static_cast<size_t>(slot) * chunks + c;
            if (hnd) {
                const int h = c / row_chunks;
                dst = ((static_cast<size_t>(page) * kv_heads + h) * page_size +
                       pos % page_size) * row_chunks + (c - h * row_chunks);
            }
            const size_t src = static_cast<size_t>(tok0 + t) * chunks + c;
            k_pool[dst] = load_streaming(k_new + src);
            v_pool[dst] = load_streaming(v_new + src);
        }
    }
}

// INT8 store (TileInfer.jl "KV cache", "INT8 cache"): one warp per (token, kv head) vector of
// D = 32 * E values.  scale = max|x| / 127 and code = rint(x / scale) clamped to [-127, 127],
// both in fp32 with round-to-nearest division, so the codes are the ones the quantiser's
// definition gives; an all-zero vector stores scale 0 and codes 0.  Codes land in the pool
// like bf16 values do ([slot][kv head][D], or [page][kv head][offset][D] for HND pools);
// scales at [page][kv head][offset].
template <int E>
__global__ void __launch_bounds__(256) store_int8_kernel(int8_t *__restrict__ k_codes,
                                                         int8_t *__restrict__ v_codes,
                                                         float *__restrict__ k_scales,
                                                         float *__restrict__ v_scales,
                                                         const __nv_bfloat16 *__restrict__ k_new,
                                                         const __nv_bfloat16 *__restrict__ v_new,
                                                         const int32_t *__restrict__ slots,
                                                         int num_tokens, int kv_heads,
                                                         int page_size, int num_slots,
                                                         uint32_t *word, bool hnd)
{
    pdl_wait();
    pdl_trigger();
    uint32_t *err = word ? word : &g_store_errors;
    constexpr int D = 32 * E;
    const int lane = threadIdx.x & 31;
    const long long vectors = static_cast<long long>(num_tokens) * kv_heads;
    const long long step = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    for (long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         w < vectors; w += step) {
        const int t = static_cast<int>(w / kv_heads);
        const int g = static_cast<int>(w - static_cast<long long>(t) * kv_heads);
        const int slot = __ldg(slots + t);
        if (slot < 0)
            continue;
        if (slot >= num_slots) {
            if (lane == 0 && g == 0)
                atomicOr(err, kErrSlotRange);
            continue;
        }
        const size_t src = static_cast<size_t>(w) * D + lane * E;
        const int page = slot / page_size;
        const size_t sidx = (static_cast<size_t>(page) * kv_heads + g) * page_size +
                            (slot - page * page_size);
        // codes: NHD [slot][kv head][D]; HND [page][kv head][offset][D] (row sidx)
        const size_t dst = (hnd ? sidx : static_cast<size_t>(slot) * kv_heads + g) * D + lane * E;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const __nv_bfloat16 *x = (which == 0 ? k_new : v_new) + src;
            float f[E];
            float m = 0.0f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                f[e] = __bfloat162float(x[e]);
                m = fmaxf(m, fabsf(f[e]));
            }
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
            int8_t *codes = (which == 0 ? k_codes : v_codes) + dst;
            if (E == 4)
                *reinterpret_cast<uint32_t *>(codes) = packed;
            else
                *reinterpret_cast<uint16_t *>(codes) = static_cast<uint16_t>(packed);
            if (lane == 0)
                (which == 0 ? k_scales : v_scales)[sidx] = scale;
        }
    }
}

// Copy-on-write: whole pages of both pools, src_pages[i] -> dst_pages[i].  chunks = 16-byte
// chunks per page (page_size * kv_heads * head_dim * 2 / 16); a grid-stride loop over
// (copy, chunk), so consecutive threads stream consecutive bytes of one page.
__global__ void __launch_bounds__(256) copy_pages_kernel(uint4 *__restrict__ k_pool,
                                                         uint4 *__restrict__ v_pool,
                                                         const int32_t *__restrict__ src_pages,
                                                         const int32_t *__restrict__ dst_pages,
                                                         int num_copies, int chunks, int num_pages,
                                                         uint32_t *word)
{
    pdl_wait();
    pdl_trigger();
    uint32_t *err = word ? word : &g_store_errors;
    const size_t total = static_cast<size_t>(num_copies) * chunks;
    const size_t step = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += step) {
        const int n = static_cast<int>(i / chunks);
        const int c = static_cast<int>(i - static_cast<size_t>(n) * chunks);
        const int src = __ldg(src_pages + n);
        const int dst = __ldg(dst_pages + n);
        if (src < 0 || src >= num_pages || dst < 0 || dst >= num_pages) {
            if (c == 0)
                atomicOr(err, kErrPageRange);
            continue;
        }
        const size_t from = static_cast<size_t>(src) * chunks + c;
        const size_t to = static_cast<size_t>(dst) * chunks + c;
        const uint4 kv = load_streaming(k_pool + from);
        const uint4 vv = load_streaming(v_pool + from);
        k_pool[to] = kv;
        v_pool[to] = vv;
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

cudaError_t launch_slot_mapping(int32_t *slots, const int32_t *block_table, int bt_stride,
                                const int32_t *context_lens, const int32_t *q_indptr,
                                int num_seqs, int num_tokens, int max_q_len, int page_size,
                                cudaStream_t stream)
{
    (void)num_tokens;
    if (num_seqs == 0)
        return cudaSuccess;
    if (q_indptr == nullptr) {
        const int threads = 128;
        return launch_pdl(slot_mapping_decode_kernel, dim3((num_seqs + threads - 1) / threads),
                          dim3(threads), 0, stream, slots, block_table, bt_stride, context_lens,
                          num_seqs, page_size, current_error_word());
    } else {
        int threads = ((max_q_len + 31) / 32) * 32;
        threads = threads < 32 ? 32 : (threads > 256 ? 256 : threads);
        return launch_pdl(slot_mapping_ragged_kernel, dim3(num_seqs), dim3(threads), 0, stream,
                          slots, block_table, bt_stride, context_lens, q_indptr, page_size,
                          current_error_word());
    }
}

cudaError_t launch_store(void *k_pool, void *v_pool, int kv_heads, int head_dim,
                         int num_slots, const void *k_new, const void *v_new,
                         const int32_t *slots, int num_tokens, cudaStream_t stream, bool hnd,
                         int page_size)
{
    if (num_tokens == 0)
        return cudaSuccess;
    const int chunks = kv_heads * head_dim * 2 / 16;
    const size_t total = static_cast<size_t>(num_tokens) * chunks;
    const int threads = 256;
    const size_t wanted = (total + threads - 1) / threads;
    const size_t cap = static_cast<size_t>(sm_count()) * 8;
    const int blocks = static_cast<int>(wanted < cap ? wanted : cap);
    return launch_pdl(store_kernel, dim3(blocks), dim3(threads), 0, stream,
                      static_cast<uint4 *>(k_pool), static_cast<uint4 *>(v_pool),
                      static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), slots,
                      num_tokens, chunks, num_slots, hnd, kv_heads, page_size,
                      current_error_word());
}

cudaError_t launch_store_boundary(void *k_pool, void *v_pool, int kv_heads, int head_dim,
                                  int page_size, int num_slots, bool hnd, const void *k_new,
                                  const void *v_new, const int32_t *block_table, int bt_stride,
                                  const int32_t *q_indptr, const int32_t *context_lens,
                                  int num_seqs, bool whole, cudaStream_t stream)
{
    if (num_seqs == 0)
        return cudaSuccess;
    const int cap = sm_count() * 8;
    const int blocks = num_seqs < cap ? num_seqs : cap;
    return launch_pdl(store_boundary_kernel, dim3(blocks), dim3(256), 0, stream,
                      static_cast<uint4 *>(k_pool), static_cast<uint4 *>(v_pool),
                      static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new),
                      block_table, bt_stride, q_indptr, context_lens, num_seqs,
                      kv_heads * head_dim * 2 / 16, kv_heads, page_size, num_slots, hnd, whole,
                      current_error_word());
}

cudaError_t launch_store_int8(void *k_codes, void *v_codes, float *k_scales, float *v_scales,
                              int kv_heads, int head_dim, int page_size, int num_slots,
                              const void *k_new, const void *v_new, const int32_t *slots,
                              int num_tokens, cudaStream_t stream, bool hnd)
{
    if (num_tokens == 0)
        return cudaSuccess;
    const long long vectors = static_cast<long long>(num_tokens) * kv_heads;
    const int threads = 256;
    const long long wanted = (vectors + 7) / 8;
    const long long cap = static_cast<long long>(sm_count()) * 8;
    const int blocks = static_cast<int>(wanted < cap ? wanted : cap);
    auto *kc = static_cast<int8_t *>(k_codes);
    auto *vc = static_cast<int8_t *>(v_codes);
    auto *kn = static_cast<const __nv_bfloat16 *>(k_new);
    auto *vn = static_cast<const __nv_bfloat16 *>(v_new);
    if (head_dim == 128)
        return launch_pdl(store_int8_kernel<4>, dim3(blocks), dim3(threads), 0, stream, kc, vc,
                          k_scales, v_scales, kn, vn, slots, num_tokens, kv_heads, page_size,
                          num_slots, current_error_word(), hnd);
    else
        return launch_pdl(store_int8_kernel<2>, dim3(blocks), dim3(threads), 0, stream, kc, vc,
                          k_scales, v_scales, kn, vn, slots, num_tokens, kv_heads, page_size,
                          num_slots, current_error_word(), hnd);
}

cudaError_t launch_copy_pages(void *k_pool, void *v_pool, int num_pages, int page_size,
                              int kv_heads, int head_dim, const int32_t *src_pages,
                              const int32_t *dst_pages, int num_copies, cudaStream_t stream)
{
    if (num_copies == 0)
        return cudaSuccess;
    const int chunks = page_size * kv_heads * head_dim * 2 / 16;
    const size_t total = static_cast<size_t>(num_copies) * chunks;
    const int threads = 256;
    const size_t wanted = (total + threads - 1) / threads;
    const size_t cap = static_cast<size_t>(sm_count()) * 8;
    const int blocks = static_cast<int>(wanted < cap ? wanted : cap);
    return launch_pdl(copy_pages_kernel, dim3(blocks), dim3(threads), 0, stream,
                      static_cast<uint4 *>(k_pool), static_cast<uint4 *>(v_pool), src_pages,
                      dst_pages, num_copies, chunks, num_pages, current_error_word());
}

cudaError_t read_and_clear_store_errors(uint32_t *flags)
{
    uint32_t zero = 0;
    cudaError_t err = cudaMemcpyFromSymbol(flags, g_store_errors, sizeof(uint32_t));
    if (err != cudaSuccess)
        return err;
    return cudaMemcpyToSymbol(g_store_errors, &zero, sizeof(uint32_t));
}

}  // namespace kvc
