// kvc_validate.cu -- opt-in deep check of block tables, context lengths and slot mappings.
//
// Integer work only.  Four checks (see include/kvc.h): lengths within a block-table row, the
// page ids a sequence reaches inside the pool, slots inside the pool, and no slot written by
// two tokens of one store (the hazard "KV Cache Management and PagedAttention", "Split shared
// blocks when a write is needed", guards against with copy-on-write).  Each check records the
// smallest offending index with atomicMin, so the verdict does not depend on thread order.
#include "kvc_launch.h"

namespace kvc {

namespace {

constexpr int kThreadsV = 256;

__global__ void validate_init_kernel(ValidateRecord *rec)
{
    if (threadIdx.x < kValidateChecks)
        rec->first_bad[threadIdx.x] = 0x7FFFFFFF;
}

// One thread per (sequence, block-table column).
__global__ void validate_tables_kernel(const int32_t *block_table, int bt_stride,
                                       const int32_t *context_lens, int num_seqs,
                                       int page_size, int num_pages, ValidateRecord *rec)
{
    const long long total = static_cast<long long>(num_seqs) * bt_stride;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
         idx < total; idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int s = static_cast<int>(idx / bt_stride);
        const int i = static_cast<int>(idx % bt_stride);
        const int ctx = context_lens[s];
        if (ctx < 0 ||
            static_cast<long long>(ctx) > static_cast<long long>(bt_stride) * page_size) {
            if (i == 0)
                atomicMin(&rec->first_bad[0], s);
            continue;
        }
        const int n_pages = (ctx + page_size - 1) / page_size;
        if (i < n_pages) {
            const int page = block_table[idx];
            if (page < 0 || page >= num_pages)
                atomicMin(&rec->first_bad[1], s);
        }
    }
}

// Pass 1 over the tokens: range check, and mark slots seen twice.
__global__ void validate_slots_mark_kernel(const int32_t *slots, int num_tokens, int num_slots,
                                           uint32_t *seen, uint32_t *dup, ValidateRecord *rec)
{
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < num_tokens;
         t += gridDim.x * blockDim.x) {
        const int slot = slots[t];
        if (slot < 0)
            continue;
        if (slot >= num_slots) {
            atomicMin(&rec->first_bad[2], t);
            continue;
        }
        const uint32_t bit = 1u << (slot & 31);
        if (atomicOr(&seen[slot >> 5], bit) & bit)
            atomicOr(&dup[slot >> 5], bit);
    }
}

// Pass 2: the smallest token whose slot was marked as written twice.
__global__ void validate_slots_dup_kernel(const int32_t *slots, int num_tokens, int num_slots,
                                          const uint32_t *dup, ValidateRecord *rec)
{
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < num_tokens;
         t += gridDim.x * blockDim.x) {
        const int slot = slots[t];
        if (slot < 0 || slot >= num_slots)
            continue;
        if (dup[slot >> 5] & (1u << (slot & 31)))
            atomicMin(&rec->first_bad[3], t);
    }
}

int grid_for(long long items)
{
    const long long blocks = (items + kThreadsV - 1) / kThreadsV;
    return static_cast<int>(blocks < 4096 ? (blocks > 0 ? blocks : 1) : 4096);
}

}  // namespace

size_t validate_workspace_bytes(long long num_slots)
{
    const size_t words = static_cast<size_t>((num_slots + 31) / 32);
    return sizeof(ValidateRecord) + 2 * words * sizeof(uint32_t);
}

cudaError_t launch_validate(const int32_t *block_table, int bt_stride, const int32_t *context_lens,
                            int num_seqs, const int32_t *slots, int num_tokens, int page_size,
                            int num_pages, void *workspace, cudaStream_t stream)
{
    const long long num_slots = static_cast<long long>(num_pages) * page_size;
    auto *rec = static_cast<ValidateRecord *>(workspace);
    uint32_t *seen = reinterpret_cast<uint32_t *>(rec + 1);
    uint32_t *dup = seen + (num_slots + 31) / 32;
    cudaError_t err =
        cudaMemsetAsync(workspace, 0, validate_workspace_bytes(num_slots), stream);
    if (err != cudaSuccess)
        return err;
    validate_init_kernel<<<1, 32, 0, stream>>>(rec);
    if (num_seqs > 0)
        validate_tables_kernel<<<grid_for(static_cast<long long>(num_seqs) * bt_stride), kThreadsV,
                                 0, stream>>>(block_table, bt_stride, context_lens, num_seqs,
                                              page_size, num_pages, rec);
    if (num_tokens > 0) {
        validate_slots_mark_kernel<<<grid_for(num_tokens), kThreadsV, 0, stream>>>(
            slots, num_tokens, static_cast<int>(num_slots), seen, dup, rec);
        validate_slots_dup_kernel<<<grid_for(num_tokens), kThreadsV, 0, stream>>>(
            slots, num_tokens, static_cast<int>(num_slots), dup, rec);
    }
    return cudaGetLastError();
}

}  // namespace kvc
