// kvc_launch.h -- host-side launchers of the kvc kernels (internal; the C ABI is kvc.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kvc {

// The device word that the calling host thread named with kvc_set_error_word, or nullptr (the
// kernels then set bits in their translation unit's own word, read by kvc_device_errors).
uint32_t *current_error_word();

// Launch with programmatic stream serialisation (see pdl_wait / pdl_trigger in kvc_device.cuh):
// the kernel may start before the previous launch on the stream has finished and waits for it
// in its first instruction.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

struct DecodeLaunch {
    const void *q;
    void *out;
    int out_f32;
    float *part_o;            // [S][Hq][n_split][D] when n_split > 1
    float *part_lse;          // [S][Hq][n_split]
    const int32_t *block_table;
    int bt_stride;
    const int32_t *context_lens;
    int num_seqs, q_heads, kv_heads, head_dim, page_size;
    int chunk, n_split;
    float scale;
    // Optional, for decode over a suffix: keys start at key_start[s] (a multiple of page
    // size), and the partials of this launch are splits split_base .. of split_stride.
    const int32_t *key_start = nullptr;
    int split_base = 0;
    int split_stride = 0;   // 0: n_split
    bool hnd = false;       // pools in the HND layout (the tensor maps follow it too)
    // Fused store (kvc_decode_store): new K / V [S][Hkv][D] and the writable pools.
    const void *k_new = nullptr, *v_new = nullptr;
    void *k_pool_w = nullptr, *v_pool_w = nullptr;
    int num_slots = 0;
};

// Decode over INT8 pages (head_dim 64 or 128): codes like a bf16 pool, scales [pages][Hkv][P].
// The positions of all (sequence, kv head) units are cut into n_ctas equal runs of 64-position
// blocks (one CTA each), whose pieces are merged by a second launch; per_unit runs one CTA per
// unit instead and writes the output directly (no workspace, no merge).
struct DecodeInt8Launch {
    const void *q;
    const float *k_scales, *v_scales;
    void *out;
    int out_f32;
    float *part_o = nullptr;      // [units + n_ctas][G][D]
    float *part_lse = nullptr;    // [units + n_ctas][G]
    void *unit_info = nullptr;    // [units] int2: first partial slot, piece count
    const int32_t *block_table;
    int bt_stride;
    const int32_t *context_lens;
    int num_seqs, q_heads, kv_heads, page_size;
    int n_ctas = 1;
    bool per_unit = false;
    float scale;
    // fused store (kvc_decode_int8_store): new K/V [S][Hkv][D] bf16 and the pools to write
    const void *k_new = nullptr, *v_new = nullptr;
    void *k_codes_w = nullptr, *v_codes_w = nullptr;
    float *k_scales_w = nullptr, *v_scales_w = nullptr;
    int num_slots = 0;
    int head_dim = 128;
    bool hnd = false;   // codes [pages][Hkv][P][D] (the tensor maps follow it too)
};
cudaError_t launch_decode_int8(const DecodeInt8Launch &l, const CUtensorMap &tmap_k,
                               const CUtensorMap &tmap_v, cudaStream_t stream);
cudaError_t read_and_clear_decode_int8_errors(uint32_t *flags);

// Grouped decode over a shared prefix: for each group, the first prefix_len[g] positions are
// the same pages for every member (the leader's block-table row lists them).
struct GroupedPrefixLaunch {
    const void *q;
    float *part_o;            // [S][Hq][split_stride][D]
    float *part_lse;          // [S][Hq][split_stride]
    const int32_t *block_table;
    int bt_stride;
    const int32_t *group_indptr;   // [num_groups + 1] into group_seqs
    const int32_t *group_seqs;
    const int32_t *prefix_len;     // [num_groups]
    int num_groups, max_rows;      // max_rows = largest group size * G (<= 64)
    int num_seqs, q_heads, kv_heads, head_dim, page_size;
    int chunk, n_split, split_stride;
    float scale;
    bool hnd = false;
    // at most this many prefix CTAs, each taking every max_prefix_ctas-th work item after its
    // first (0: one CTA per item)
    int max_prefix_ctas = 0;
};

struct AppendLaunch {
    const void *q;
    void *out;
    int out_f32;
    const int32_t *block_table;
    int bt_stride;
    const int32_t *q_indptr;
    const int32_t *context_lens;
    int num_seqs, num_tokens, max_q_len, q_heads, kv_heads, head_dim, page_size;
    float scale;
    bool hnd = false;
    // kvc_append_store: the chunk's K/V come from k_new / v_new (tmap_kn / tmap_vn) and the
    // kernel writes them to the pools (k_pool_w / v_pool_w), except the boundary tokens
    // launch_store_boundary wrote before.
    bool fused = false;
    void *k_pool_w = nullptr, *v_pool_w = nullptr;
    int num_pages = 0;   // pages of the pools (fused: a page id outside them is skipped)
};

// kvc_append_int8: AppendLaunch over INT8 pages (head_dim 64 or 128) plus the scale arrays.
struct AppendInt8Launch {
    void *out;
    int out_f32;
    const float *k_scales, *v_scales;   // [num_pages][kv_heads][page_size]
    const int32_t *block_table;
    int bt_stride;
    const int32_t *q_indptr;
    const int32_t *context_lens;
    int num_seqs, num_tokens, max_q_len, q_heads, kv_heads, page_size;
    float scale;
    int head_dim = 128;
    bool hnd = false;   // codes [pages][Hkv][P][D] (the tensor maps follow it too)
};

// kvc_validate: the smallest offending index of each check (INT32_MAX when it passed), then two
// bitmaps over the pool's slots.
constexpr int kValidateChecks = 4;
struct ValidateRecord {
    int first_bad[kValidateChecks];
};
size_t validate_workspace_bytes(long long num_slots);
cudaError_t launch_validate(const int32_t *block_table, int bt_stride, const int32_t *context_lens,
                            int num_seqs, const int32_t *slots, int num_tokens, int page_size,
                            int num_pages, void *workspace, cudaStream_t stream);

// Each returns cudaSuccess or the launch error.
cudaError_t launch_slot_mapping(int32_t *slots, const int32_t *block_table, int bt_stride,
                                const int32_t *context_lens, const int32_t *q_indptr,
                                int num_seqs, int num_tokens, int max_q_len, int page_size,
                                cudaStream_t stream);
cudaError_t launch_store(void *k_pool, void *v_pool, int kv_heads, int head_dim,
                         int num_slots, const void *k_new, const void *v_new,
                         const int32_t *slots, int num_tokens, cudaStream_t stream,
                         bool hnd = false, int page_size = 1);
cudaError_t launch_store_int8(void *k_codes, void *v_codes, float *k_scales, float *v_scales,
                              int kv_heads, int head_dim, int page_size, int num_slots,
                              const void *k_new, const void *v_new, const int32_t *slots,
                              int num_tokens, cudaStream_t stream, bool hnd = false);
cudaError_t launch_copy_pages(void *k_pool, void *v_pool, int num_pages, int page_size,
                              int kv_heads, int head_dim, const int32_t *src_pages,
                              const int32_t *dst_pages, int num_copies, cudaStream_t stream);
cudaError_t launch_decode(const DecodeLaunch &a, const CUtensorMap &tmap_k,
                          const CUtensorMap &tmap_v, cudaStream_t stream);
cudaError_t launch_merge(void *out, int out_f32, const float *part_o, const float *part_lse,
                         int rows, int n_split, int head_dim, float *lse_out,
                         cudaStream_t stream);
// Grouped decode: sets key_start to 0, then each group's members' key_start to the group's
// prefix length (one block; the grouped grid marks the empty prefix partials itself).
cudaError_t launch_grouped_setup(int32_t *key_start, const int32_t *group_indptr,
                                 const int32_t *group_seqs, const int32_t *prefix_len,
                                 int num_groups, int num_seqs, int page_size, int bt_stride,
                                 cudaStream_t stream);
// Groups from block tables (adjacent sequences agreeing on leading shareable pages), one CTA:
// group_indptr[num_seqs / 2 + 1], group_seqs[num_seqs], prefix_len[num_seqs / 2], num_groups[1].
cudaError_t launch_group_detect(const int32_t *block_table, int bt_stride,
                                const int32_t *context_lens, int num_seqs, int page_size,
                                int max_members, int32_t *group_indptr, int32_t *group_seqs,
                                int32_t *prefix_len, int32_t *num_groups, cudaStream_t stream);
// The prefix CTAs of `p` and the suffix decode of `l` (key_start set, partials after the
// prefix splits) in one grid.
cudaError_t launch_grouped_decode(const GroupedPrefixLaunch &p, const DecodeLaunch &l,
                                  const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                                  cudaStream_t stream);
// tmap_q views q as [T][kv_heads][G][head_dim] with 128-row boxes; tmap_kn / tmap_vn (fused
// only) view k_new / v_new as {head_dim, kv head, token} with {64, 1, page_size} boxes.
cudaError_t launch_append_tc(const AppendLaunch &a, const CUtensorMap &tmap_q,
                             const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                             cudaStream_t stream, const CUtensorMap *tmap_kn = nullptr,
                             const CUtensorMap *tmap_vn = nullptr);
// The new tokens that share a page with cached positions (the chunk's first page when
// (ctx - q_len) % page_size != 0), stored at their slots from the block table.
cudaError_t launch_store_boundary(void *k_pool, void *v_pool, int kv_heads, int head_dim,
                                  int page_size, int num_slots, bool hnd, const void *k_new,
                                  const void *v_new, const int32_t *block_table, int bt_stride,
                                  const int32_t *q_indptr, const int32_t *context_lens,
                                  int num_seqs, bool whole, cudaStream_t stream);
// tmap_q as for launch_append_tc; tmap_k / tmap_v are the INT8 page maps (one box per page).
cudaError_t launch_append_int8(const AppendInt8Launch &a, const CUtensorMap &tmap_q,
                               const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                               cudaStream_t stream);

// Device error words, one per translation unit that owns bounded waits.
cudaError_t read_and_clear_decode_errors(uint32_t *flags);
// One CTA whose bounded wait runs out (about a second): sets kErrSelftestWait.
cudaError_t launch_selftest_wait(cudaStream_t stream);
cudaError_t read_and_clear_store_errors(uint32_t *flags);
cudaError_t read_and_clear_append_tc_errors(uint32_t *flags);
cudaError_t read_and_clear_grouped_errors(uint32_t *flags);
cudaError_t read_and_clear_append_int8_errors(uint32_t *flags);

// Record a failure reason for kvc_last_error() from another translation unit.
int set_last_error(int status, const char *message);

// Stage geometry shared by the decode and append pipelines: a stage holds kStageKeys
// positions of one kv head as whole pages, each page stored [half][page_size rows][64 columns]
// with 128-byte swizzle (one TMA box per page).
constexpr int kStageKeys = 64;   // positions per pipeline stage

}  // namespace kvc
