// kvc_append_items.cuh -- the work items of the append kernels and the walker over them.
//
// The rows of one (sequence, kv head) are its (new token, query head of the group) pairs,
// token-major, in tiles of 128; a work item is a pair of consecutive tiles of one (sequence,
// kv head).  A persistent CTA walks items c, c + grid, ...; every role of the CTA walks the
// same items in the same order.  Args is the kernel's argument struct; it provides q_indptr,
// context_lens, bt_stride, page_size, group, kv_heads, pairs_per_seq and num_items.
#pragma once

#include <stdint.h>

#include "kvc_device.cuh"

namespace kvc {
namespace append {

constexpr int kM = 128;    // rows per tile
constexpr int kBN = 128;   // positions per K or V stage

// One work item: tiles 2 tp and 2 tp + 1 of one (sequence, kv head).
struct Item {
    int s, kvh, tp;
    int tok0, q_len, ctx, rows, row_begin;   // row_begin: first row of tile 2 tp
    bool has_b;                              // tile 2 tp + 1 exists
    int n_keys, n_blocks;                    // positions the item's later tile sees
    bool over;                               // context_lens[s] exceeded the block-table row
};

// The fields of item `it` from its sequence's query offsets and context length (no loads).
template <class Args>
__device__ __forceinline__ bool make_item(const Args &a, int it, int tok0, int tok1, int ctx,
                                          Item &x, uint32_t *err)
{
    x.tp = it % a.pairs_per_seq;
    const int rest = it / a.pairs_per_seq;
    x.kvh = rest % a.kv_heads;
    x.s = rest / a.kv_heads;
    x.tok0 = tok0;
    x.q_len = tok1 - tok0;
    x.ctx = ctx;
    x.over = x.ctx > a.bt_stride * a.page_size;
    if (x.over) {
        if (threadIdx.x == 0)
            atomicOr(err, kErrContextRange);
        x.ctx = a.bt_stride * a.page_size;
    }
    x.rows = x.q_len * a.group;
    x.row_begin = x.tp * 2 * kM;
    if (x.row_begin >= x.rows)
        return false;
    x.has_b = x.row_begin + kM < x.rows;
    const int row_last = min(x.rows, x.row_begin + 2 * kM) - 1;
    x.n_keys = min(x.ctx, x.ctx - x.q_len + row_last / a.group + 1);
    if (x.n_keys <= 0)
        return false;
    x.n_blocks = (x.n_keys + kBN - 1) / kBN;
    return true;
}

template <class Args>
__device__ __forceinline__ int seq_of(const Args &a, int it)
{
    return it / a.pairs_per_seq / a.kv_heads;
}

// Walks this CTA's items: it = blockIdx.x, blockIdx.x + gridDim.x, ..., skipping empty ones.
// A global load under a full memory pipe takes microseconds, so the metadata of the next
// item index is requested one item ahead (its registers are read only at the next step).
struct Walker {
    int it;
    bool done;
    Item x;
    int pit;                  // index whose metadata is in flight in p_*
    int p_tok0, p_tok1, p_ctx;
    template <class Args>
    __device__ __forceinline__ void prefetch(const Args &a, int idx)
    {
        pit = idx;
        if (idx < a.num_items) {
            const int s = seq_of(a, idx);
            p_tok0 = a.q_indptr[s];
            p_tok1 = a.q_indptr[s + 1];
            p_ctx = a.context_lens[s];
        }
    }
    template <class Args>
    __device__ __forceinline__ void next(const Args &a, uint32_t *err)
    {
        for (;;) {
            it += gridDim.x;
            if (it >= a.num_items) {
                done = true;
                return;
            }
            int tok0, tok1, ctx;
            if (it == pit) {
                tok0 = p_tok0;
                tok1 = p_tok1;
                ctx = p_ctx;
            } else {
                const int s = seq_of(a, it);
                tok0 = a.q_indptr[s];
                tok1 = a.q_indptr[s + 1];
                ctx = a.context_lens[s];
            }
            if (make_item(a, it, tok0, tok1, ctx, x, err))
                break;
        }
        prefetch(a, it + gridDim.x);
    }
    template <class Args>
    __device__ __forceinline__ void start(const Args &a, uint32_t *err)
    {
        it = static_cast<int>(blockIdx.x) - static_cast<int>(gridDim.x);
        done = false;
        pit = -1;
        next(a, err);
    }
};

}  // namespace append
}  // namespace kvc
