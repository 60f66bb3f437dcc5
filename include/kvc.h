/*
 * kvc.h -- paged KV-cache store and paged attention for NVIDIA GB300 (sm_103a).
 *
 * A KV cache kept in fixed-size pages, addressed through per-sequence block tables:
 *   TileInfer.jl "KV cache", sections "Pages and block tables" and "Growing, rolling back,
 *   releasing"; "KV Cache Management and PagedAttention", sections "Connect token order to
 *   storage locations", "Compute attention over scattered KV" and "Share common KV across
 *   responses"; Quail "KV", sections "Paged KV", "KV rewind" and "Prefix sharing".
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 * Pools.  One K pool and one V pool per layer, each bf16 [num_pages][page_size][kv_heads]
 *   [head_dim], row-major (the (position, kv head) vector is head_dim contiguous values).
 *   Viewed by slot it is [num_pages * page_size][kv_heads][head_dim].  pool.layout = KVC_HND
 *   selects [num_pages][kv_heads][page_size][head_dim] instead (see kvc_layout), for bf16 and
 *   INT8 pages alike.
 * Address rule.  Position p (0-based) of sequence s lives in page block_table[s][p /
 *   page_size] at offset p % page_size; its slot is page * page_size + offset.
 * Block table.  int32 [num_seqs][bt_stride], row-major.  Entries past a sequence's last
 *   page are never read (the caller may zero-pad rows to a fixed width, e.g. a multiple of
 *   16, so that a captured CUDA graph stays valid as sequences grow; page 0 in the padding
 *   is harmless).  Several rows may list the same pages (a shared prefix).
 * context_lens[s].  Number of positions of sequence s including the new token(s); the
 *   newest token attends to its own key and value, so its K/V must be stored first.
 * GQA.  q_heads = G * kv_heads; q head h reads kv head h / G.
 * Scale.  Scores are q.k * scale; scale <= 0 selects 1/sqrt(head_dim).
 * Memory.  Every pointer argument named *pool, q, k_new, v_new, out, block_table,
 *   context_lens, q_indptr, slot_mapping, partial_*, workspace is a DEVICE pointer owned by
 *   the caller (kvc_decode's q, tables and out, kvc_merge's out, kvc_store's k_new / v_new
 *   and kvc_slot_mapping's tables may also be pinned host memory mapped at its host
 *   address, see each call).
 *   The library allocates no memory, holds no pointer after a call returns,
 *   and never synchronises: each call only enqueues kernels on `stream` (a cudaStream_t;
 *   NULL is the legacy default stream).  Device arrays are not read on the host, so per-step
 *   values may change between replays of a captured graph.
 * Alignment.  bf16 tensors and pools must be 16-byte aligned (TMA and 16-byte vector
 *   accesses); fp32 partials 16-byte aligned.
 * Errors.  Scalars are checked on the host before anything is enqueued; a bad call returns
 *   a status and enqueues nothing.  Device-side contents (page ids, slots, lengths) are
 *   trusted: out-of-range values there are caller errors (page ids must be < num_pages,
 *   context_lens[s] <= bt_stride * page_size).  kvc_last_error() gives a one-line reason
 *   for the last failing call on the calling thread.
 * Supported shapes.  head_dim 64 or 128; page_size 16, 32 or 64; G = q_heads / kv_heads
 *   in {1, 2, 4, 8}; num_pages * page_size < 2^31.  Others return KVC_ERR_UNSUPPORTED.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvc_status {
    KVC_OK = 0,
    KVC_ERR_INVALID_ARG = 1,  /* null pointer, negative size, misaligned pointer ...      */
    KVC_ERR_UNSUPPORTED = 2,  /* shape outside the supported set above                   */
    KVC_ERR_WORKSPACE = 3,    /* workspace missing or smaller than the plan requires      */
    KVC_ERR_CUDA = 4,         /* a CUDA call failed (launch, tensor-map encode, ...)      */
    KVC_ERR_DEVICE = 5,       /* a kernel gave up a bounded wait (see kvc_device_errors)  */
    KVC_ERR_OUT_OF_RANGE = 6  /* kvc_validate found a bad table entry, slot or length       */
} kvc_status;

typedef enum kvc_dtype {
    KVC_BF16 = 0,             /* bf16, rounded to nearest even from the fp32 accumulator */
    KVC_F32 = 1
} kvc_dtype;

typedef enum kvc_layout {
    KVC_NHD = 0,              /* [num_pages][page_size][kv_heads][head_dim] (default)       */
    KVC_HND = 1               /* [num_pages][kv_heads][page_size][head_dim]: one contiguous
                                 block per (page, kv head) -- TileInfer.jl "KV cache", "Pages
                                 and block tables", its (head_dim, page_size, kv_heads,
                                 num_pages) column-major array; bf16 pools only             */
} kvc_layout;

typedef struct kvc_pool_desc {
    int32_t num_pages;
    int32_t page_size;        /* positions per page                                       */
    int32_t kv_heads;
    int32_t head_dim;
    int32_t layout;           /* kvc_layout; slots (page * page_size + offset) mean the same
                                 positions in either layout                                 */
} kvc_pool_desc;

/* Human-readable name of a status, and the reason for the last failure on this thread. */
const char *kvc_status_string(kvc_status status);
const char *kvc_last_error(void);

/*
 * kvc_slot_mapping -- slot of every new token (TileInfer.jl "KV cache", "Pages and block
 * tables": before a step, each new token's slot is computed from the block table).
 *
 * New token i of sequence s (0 <= i < q_len_s, q_len_s = q_indptr[s+1] - q_indptr[s]) is
 * at position context_lens[s] - q_len_s + i; slot_mapping[q_indptr[s] + i] receives its
 * slot.  q_indptr == NULL means one new token per sequence (decode): token s belongs to
 * sequence s and num_tokens must equal num_seqs.  A position below zero (context_lens[s] <
 * q_len_s) yields slot -1.  Integer arithmetic only: bit-exact.
 *   slot_mapping  int32 [num_tokens]        (out)
 *   block_table   int32 [num_seqs][bt_stride]
 *   context_lens  int32 [num_seqs]
 *   q_indptr      int32 [num_seqs + 1] or NULL
 * block_table, context_lens and q_indptr may also be pinned host memory that the device
 * reaches at its host address (the kernel reads the few entries it needs across the host
 * link, so a step's tables need not be copied first for this call); any other host pointer:
 * KVC_ERR_INVALID_ARG, nothing enqueued.
 *   max_q_len     host upper bound on q_len_s (sizes the launch; 1 when q_indptr is NULL)
 */
kvc_status kvc_slot_mapping(int32_t *slot_mapping, const int32_t *block_table,
                            int32_t bt_stride, const int32_t *context_lens,
                            const int32_t *q_indptr, int32_t num_seqs, int32_t num_tokens,
                            int32_t max_q_len, int32_t page_size, void *stream);

/*
 * kvc_store -- write each new token's key and value at its slot (TileInfer.jl "KV cache",
 * "Pages and block tables": the step writes the new keys and values at their slots;
 * "KV Cache Management and PagedAttention", "Grow the allocation as generation proceeds").
 *
 * k_pool[slot_mapping[t]][g][:] = k_new[t][g][:] and likewise for V, for every kv head g.
 * A raw 16-bit copy: NaN payloads and signed zeros are kept.  slot_mapping[t] < 0 skips
 * token t (padding).  Slots must be < num_pages * page_size and distinct within one call
 * (two writers of one slot is the race copy-on-write exists to prevent).
 *   k_new, v_new  bf16 [num_tokens][kv_heads][head_dim]; device memory, or pinned host
 *                 memory that the device reaches at its host address (the kernel reads the
 *                 step's new keys and values across the host link); any other host pointer:
 *                 KVC_ERR_INVALID_ARG, nothing enqueued.
 */
kvc_status kvc_store(void *k_pool, void *v_pool, kvc_pool_desc pool, const void *k_new,
                     const void *v_new, const int32_t *slot_mapping, int32_t num_tokens,
                     void *stream);

/*
 * kvc_decode -- paged attention for one new token per sequence, GQA, reading K/V in place
 * from scattered pages with no gather copy ("KV Cache Management and PagedAttention",
 * "Compute attention over scattered KV"):
 *   out[s][h] = softmax_p( q[s][h] . K_s[p][h/G] * scale ) . V_s[p][h/G],  p < ctx_s,
 * where K_s[p] is the pool entry the address rule gives for position p of sequence s.
 * ctx_s = 0 yields out = 0.
 *
 * Split-K ("flash decoding"): with more than one split, the positions of each sequence are
 * cut into consecutive chunks of `chunk` positions (kvc_decode_plan); each chunk writes an
 * fp32 partial, normalised over its own keys, and its log-sum-exp into the workspace, and
 * kvc_merge (enqueued by this call) combines them.  The result does not depend on the
 * split count beyond fp32 rounding.
 *   out           [num_seqs][q_heads][head_dim], out_dtype KVC_BF16 or KVC_F32.  Device
 *                 memory, or pinned host memory that the device reaches at its host
 *                 address (cudaHostAlloc / cudaHostRegister on a UVA system): the kernel
 *                 that finishes each row then writes it straight to host memory, so the
 *                 result is on the host when the call's work completes, with no copy to
 *                 enqueue.  Any other host pointer: KVC_ERR_INVALID_ARG, nothing enqueued.
 *   q             bf16 [num_seqs][q_heads][head_dim]
 *   q, block_table, context_lens may also be pinned host memory mapped at its host address:
 *                 the kernels read them across the host link (each CTA its query rows and
 *                 page ids), so a step's inputs need no copy first.
 *   max_ctx       host upper bound on every context_lens[s] (sizes the launch)
 *   num_splits    0 = choose automatically, 1 = no split, n > 1 = at most n chunks
 *   workspace     device scratch of at least kvc_decode_plan(...)'s workspace bytes when
 *                 the plan has more than one split (may be NULL otherwise).  Layout:
 *                 partial_o fp32 [num_seqs][q_heads][splits][head_dim] at offset 0, then
 *                 partial_lse fp32 [num_seqs][q_heads][splits] at the 256-byte-aligned
 *                 offset that follows.  Splits that hold no position get lse = -inf and
 *                 an unwritten partial_o.
 */
kvc_status kvc_decode(void *out, int32_t out_dtype, const void *q, const void *k_pool,
                      const void *v_pool, kvc_pool_desc pool, const int32_t *block_table,
                      int32_t bt_stride, const int32_t *context_lens, int32_t num_seqs,
                      int32_t max_ctx, int32_t q_heads, float scale, int32_t num_splits,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * kvc_decode_store -- kvc_slot_mapping (one new token per sequence) + kvc_store + kvc_decode
 * in one call ("KV Cache Management and PagedAttention", "Grow the allocation as generation
 * proceeds" and "Compute attention over scattered KV"; TileInfer.jl "KV cache", "Pages and
 * block tables": the step writes the new key and value at their slot, and TileInfer does that
 * inside the kernel that prepares attention's inputs): the decode CTA whose chunk ends at
 * sequence s's newest position (ctx_s - 1) writes that token's key and value (k_new[s],
 * v_new[s], bf16 [num_seqs][kv_heads][head_dim])
 * for its kv head at the slot block_table[s][(ctx_s - 1) / page_size] * page_size +
 * (ctx_s - 1) % page_size, before its own copy of that page, and the attention reads it
 * there.  The pools end exactly as the three calls leave them and so does out (the same
 * kernels read the same values in the same order).  Sequences with ctx_s = 0 store nothing;
 * a slot past the pool is skipped and flagged (kvc_device_errors), as in kvc_store.  Two
 * launches (decode, and merge when split) instead of four.  Arguments as kvc_decode, plus
 * k_new / v_new (device or pinned host memory, 16-byte aligned); the pools are written.
 */
kvc_status kvc_decode_store(void *out, int32_t out_dtype, const void *q, const void *k_new,
                            const void *v_new, void *k_pool, void *v_pool, kvc_pool_desc pool,
                            const int32_t *block_table, int32_t bt_stride,
                            const int32_t *context_lens, int32_t num_seqs, int32_t max_ctx,
                            int32_t q_heads, float scale, int32_t num_splits, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * kvc_decode_plan -- the split plan kvc_decode will use for these scalars: the number of
 * splits (>= 1), the chunk length in positions (a multiple of 64 and of page_size; equal
 * to the padded max_ctx when splits == 1) and the workspace bytes it needs (0 when
 * splits == 1).  Any output pointer may be NULL.
 */
kvc_status kvc_decode_plan(int32_t num_seqs, int32_t q_heads, kvc_pool_desc pool,
                           int32_t max_ctx, int32_t num_splits, int32_t *splits_out,
                           int32_t *chunk_out, size_t *workspace_bytes_out);

/*
 * kvc_shared_prefix_groups -- find the groups for kvc_decode_shared_prefix from the block
 * tables alone (an opt-in prepass; the caller may build the groups itself instead).  Shared
 * pages are those "KV Cache Management and PagedAttention", "Share common KV across
 * responses" and Quail "KV", "Prefix sharing" / "The sharing plan" put in several block
 * tables; this finds them again by comparing adjacent tables.
 * Sequences s - 1 and s are linked when their block-table rows agree on at least the first
 * page both can share; a sequence can share only whole pages before the page of its last
 * position (its newest token goes to a page of its own): floor((ctx - 1) / page_size) pages,
 * at most bt_stride.  A group is a maximal run of linked sequences, cut into consecutive
 * chunks of at most max_members (2 .. 64; kvc_decode_shared_prefix takes members *
 * q_heads / kv_heads <= 64); a chunk of one sequence is no group.  A group's prefix is the
 * smallest agreement between adjacent members, in positions (pages * page_size).  Integer
 * work, one CTA; the result is exact (tested against the oracle's groups).
 *   block_table    int32 [num_seqs][bt_stride];  context_lens int32 [num_seqs] (device)
 *   group_indptr   int32 [num_seqs / 2 + 1] (out, device): members of group g are
 *                  group_seqs[group_indptr[g] .. group_indptr[g + 1])
 *   group_seqs     int32 [num_seqs] (out, device), ascending within and across groups
 *   prefix_len     int32 [num_seqs / 2] (out, device)
 *   num_groups     int32 [1] (out, device): the number of groups found
 * Slots g >= *num_groups of the capacity num_seqs / 2 are written as empty groups with a
 * zero prefix, so the outputs can go to kvc_decode_shared_prefix with num_groups =
 * num_seqs / 2 and max_prefix_len = max_ctx without reading the count back (empty groups
 * cost a CTA that exits at once), or with the count read back for a tighter launch.
 */
kvc_status kvc_shared_prefix_groups(const int32_t *block_table, int32_t bt_stride,
                                    const int32_t *context_lens, int32_t num_seqs,
                                    int32_t page_size, int32_t max_members,
                                    int32_t *group_indptr, int32_t *group_seqs,
                                    int32_t *prefix_len, int32_t *num_groups, void *stream);

/*
 * kvc_decode_shared_prefix -- kvc_decode for batches in which groups of sequences begin with
 * the same physical pages ("KV Cache Management and PagedAttention", "Share common KV across
 * responses": several block tables point at one copy of the common KV; each response still
 * attends with its own query over its own context; Quail "KV", "Prefix sharing").
 *
 * The result is exactly kvc_decode's (up to fp32 rounding); the shared pages are read once
 * per group instead of once per member.  Group g's members are the sequences
 * group_seqs[group_indptr[g] .. group_indptr[g+1]); every member's block table lists the same
 * first prefix_len[g] / page_size pages (the first member's row is the one read) and every
 * member's context_lens is at least prefix_len[g] (rounded down to whole pages).  A sequence
 * may belong to at most one group; sequences in no group are decoded over their whole context.
 *   group_indptr    int32 [num_groups + 1] (device)
 *   group_seqs      int32 [group_indptr[num_groups]] sequence indices (device)
 *   prefix_len      int32 [num_groups] shared positions (device)
 *   max_group_size  host bound on members per group; max_group_size * G must be <= 64
 *   max_prefix_len  host bound on prefix_len
 *   workspace       kvc_decode_shared_prefix_plan(...) bytes (required), 16-byte aligned
 * The other arguments are kvc_decode's.  Three kernels are enqueued: a set-up pass (each
 * sequence's prefix end), one grid of the prefix partials (one CTA per prefix chunk, kv head
 * and group) followed by the suffix partials (a decode CTA per kv head and sequence, from its
 * prefix end), and the log-sum-exp merge.  Empty group slots cost a CTA that exits after
 * reading its group's bounds.
 */
kvc_status kvc_decode_shared_prefix(void *out, int32_t out_dtype, const void *q,
                                    const void *k_pool, const void *v_pool, kvc_pool_desc pool,
                                    const int32_t *block_table, int32_t bt_stride,
                                    const int32_t *context_lens, int32_t num_seqs,
                                    int32_t max_ctx, int32_t q_heads, float scale,
                                    const int32_t *group_indptr, const int32_t *group_seqs,
                                    const int32_t *prefix_len, int32_t num_groups,
                                    int32_t max_group_size, int32_t max_prefix_len,
                                    void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes kvc_decode_shared_prefix needs for these scalars. */
kvc_status kvc_decode_shared_prefix_plan(int32_t num_seqs, int32_t q_heads, kvc_pool_desc pool,
                                         int32_t max_ctx, int32_t num_groups,
                                         int32_t max_prefix_len, size_t *workspace_bytes_out);

/*
 * kvc_decode_noalloc -- kvc_decode for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point; it exists for callers of this library
 * that are handed only their input and output buffers: an operator plugged into an
 * inference engine that planned every byte of device memory when it started, or a serving
 * loop that must not call cudaMalloc while it runs, because that call can synchronise the
 * whole device and take an unbounded time.  Such a caller cannot provide kvc_decode's
 * workspace.  Here the split partials go instead to scratch memory inside the library: one
 * statically sized device array of KVC_NOALLOC_SCRATCH_BYTES, which every GPU that loads the
 * library holds until the process exits.  Nothing is allocated by the call.
 *
 * Arguments and result are those of kvc_decode without the workspace.  A split plan that
 * needs more than KVC_NOALLOC_SCRATCH_BYTES of partials (see kvc_decode_plan) is rejected
 * with KVC_ERR_WORKSPACE and nothing is enqueued: ask for fewer splits, or use kvc_decode
 * with a workspace of your own.  The first call on each device (the current device) looks
 * up where the scratch array lives on that device; make that first call before any stream
 * capture.  The address is kept with the id of the context it was found in; after a device
 * reset (cudaDeviceReset) the next call finds a new context and looks it up again, so make
 * that call outside a capture too.  Every call uses the same array, which keeps what the last call wrote; nothing
 * in it has to start at zero, but two calls whose kernels overlap on the GPU (launched on
 * different streams with no ordering between them) race on it, so the caller must order them.
 */
#define KVC_NOALLOC_SCRATCH_BYTES (8u << 20)

kvc_status kvc_decode_noalloc(void *out, int32_t out_dtype, const void *q,
                              const void *k_pool, const void *v_pool, kvc_pool_desc pool,
                              const int32_t *block_table, int32_t bt_stride,
                              const int32_t *context_lens, int32_t num_seqs, int32_t max_ctx,
                              int32_t q_heads, float scale, int32_t num_splits, void *stream);

/*
 * kvc_merge -- combine split partials by log-sum-exp.  For every row r:
 *   M = max_j lse[r][j];  w_j = exp(lse[r][j] - M);
 *   out[r] = sum_j w_j partial_o[r][j] / sum_j w_j;   lse_out[r] = M + log(sum_j w_j).
 * Splits with lse = -inf hold no key: their partial_o is not used (the first few splits'
 * partials are loaded with the lse values, so partial_o must span every split).  A row whose
 * splits are all empty gets out = 0 and lse_out = -inf.  out may be pinned host memory, as for
 * kvc_decode.  (The pages leave partitioning and combining
 * inside the kernel open -- "KV Cache Management and PagedAttention", "Compute attention
 * over scattered KV"; this is the plain combination of softmax-normalised pieces.)
 *   partial_o    fp32 [rows][num_splits][head_dim]
 *   partial_lse  fp32 [rows][num_splits]
 *   out          [rows][head_dim], out_dtype KVC_BF16 or KVC_F32
 *   lse_out      fp32 [rows] or NULL (natural log)
 */
kvc_status kvc_merge(void *out, int32_t out_dtype, const float *partial_o,
                     const float *partial_lse, int32_t rows, int32_t num_splits,
                     int32_t head_dim, float *lse_out, void *stream);

/*
 * kvc_append -- causal chunked prefill of new tokens over an already-cached prefix, the
 * kernel behind KV rewind and shared-prefix reuse (Quail "KV", "KV rewind" and "Prefix
 * sharing"; TileInfer.jl "KV cache", "Growing, rolling back, releasing" and "Prefix reuse
 * in chat").  New token i of sequence s sits at position c_i = ctx_s - q_len_s + i and
 *   out[t][h] = softmax_{p <= c_i}( q[t][h] . K_s[p][h/G] * scale ) . V_s[p][h/G]
 * with t = q_indptr[s] + i.  The new tokens' K/V must already be in the pools (kvc_store).
 *   q, out        [num_tokens][q_heads][head_dim]; q bf16, out per out_dtype
 *   q_indptr      int32 [num_seqs + 1], q_indptr[0] = 0, q_indptr[num_seqs] = num_tokens
 *   max_q_len     host upper bound on every q_len_s;  max_ctx likewise for context_lens
 */
kvc_status kvc_append(void *out, int32_t out_dtype, const void *q, const void *k_pool,
                      const void *v_pool, kvc_pool_desc pool, const int32_t *block_table,
                      int32_t bt_stride, const int32_t *q_indptr,
                      const int32_t *context_lens, int32_t num_seqs, int32_t num_tokens,
                      int32_t max_q_len, int32_t max_ctx, int32_t q_heads, float scale,
                      void *stream);

/*
 * kvc_append_store -- kvc_slot_mapping + kvc_store + kvc_append in one pass over the chunk
 * (TileInfer.jl "KV cache": the store is fused into the kernel that stages K/V for attention).
 * Stores every new token's k_new / v_new row at the slot its position gets from the block
 * table (exactly what kvc_store with kvc_slot_mapping's slots writes), and returns kvc_append's
 * output for the same arguments.  The chunk's K/V are read once from k_new / v_new: the pages
 * that hold only new tokens are attended from there and written to the pools by the attention
 * kernel itself; the new tokens that share a page with cached positions (the chunk's first
 * page when ctx - q_len is not a multiple of page_size) are stored by a small kernel first.
 * With page_size >= 64 that page holds most of a short chunk and the fused read gains nothing:
 * there the small kernel stores the whole chunk and the plain append follows (same results).
 *   k_new, v_new   bf16 [num_tokens][kv_heads][head_dim], row t = token t of q (q_indptr)
 *   k_pool, v_pool written (the new tokens' slots only) and read
 * Other arguments as kvc_append.  A token whose position is negative (context_lens[s] <
 * q_len_s) is not stored.  A context longer than its block-table row (context_lens[s] >
 * bt_stride * page_size) is an error the pools survive as they do kvc_slot_mapping +
 * kvc_store: the chunk's tokens the row covers are stored at their slots, the others are
 * skipped, and the device error word (kvc_device_errors) gets 1 << 7; that sequence's output
 * is undefined.  A block-table entry outside the pool (a page id < 0 or >= pool.num_pages) is
 * likewise skipped for the tokens it would hold, as kvc_store skips a slot past the pool, with
 * 1 << 6; that sequence's output is undefined.  Two launches on `stream`.
 */
kvc_status kvc_append_store(void *out, int32_t out_dtype, const void *q, const void *k_new,
                            const void *v_new, void *k_pool, void *v_pool, kvc_pool_desc pool,
                            const int32_t *block_table, int32_t bt_stride,
                            const int32_t *q_indptr, const int32_t *context_lens,
                            int32_t num_seqs, int32_t num_tokens, int32_t max_q_len,
                            int32_t max_ctx, int32_t q_heads, float scale, void *stream);

/*
 * kvc_device_errors -- read and clear the library's own device-side error words.  Kernels
 * bound every wait (about one second); a wait that runs out sets a bit and the kernel returns
 * early, leaving its outputs undefined; range checks (a slot past the pool, a context longer
 * than its block-table row, ...) set theirs and skip the offending token.  The bits of calls
 * made while no caller word is set (kvc_set_error_word) land in these words, one per kernel
 * family in each process, on the current device: calls from several threads or streams share
 * them, and this read (which synchronises with the device) clears them for all.  *flags_out
 * = 0 when nothing was flagged since the last read.
 */
kvc_status kvc_device_errors(uint32_t *flags_out);

/*
 * kvc_set_error_word -- error reporting per caller.  Every later call from the calling host
 * thread passes `device_word` to its kernels, which OR their error bits (the bits of
 * kvc_device_errors) into it instead of into the library's own words; NULL restores those.
 * The word belongs to the caller: device memory (or pinned host memory mapped at its host
 * address) that stays valid while the calls that were given it run.  The library never reads
 * or clears it -- the caller zeroes it and reads it back on its own stream (a captured CUDA
 * graph keeps the word it was captured with).  Two callers with words of their own, on
 * different threads or streams, never see each other's bits.  Host-side argument checks still
 * return their status at once.  Returns KVC_ERR_INVALID_ARG for a word not 4-byte aligned.
 * (No counterpart on the pages: it scopes this library's failure reports.)
 */
kvc_status kvc_set_error_word(uint32_t *device_word);

/*
 * kvc_selftest_wait -- a diagnostic of the failure path every kernel shares: one CTA waits on
 * an mbarrier phase that nothing completes, with the same bounded wait the kernels use; after
 * about a second it gives up, sets bit 1 << 12 of the device error word (kvc_device_errors)
 * and returns.  Nothing faults or hangs, and later calls run as usual.
 */
kvc_status kvc_selftest_wait(void *stream);

/*
 * INT8 pages (TileInfer.jl "KV cache", section "INT8 cache": the pools hold int8 codes with
 * one fp32 scale per cached vector -- one kv head at one position -- x ~ scale * code,
 * symmetric, scale = max|x| / 127, quantised once when the position is written; attention
 * does not dequantise: a key's scale multiplies its score, a value's scale its probability
 * before the PV product).  132 bytes per vector at head_dim 128 instead of 256.
 *   k_codes, v_codes   int8 [num_pages][page_size][kv_heads][head_dim] (the bf16 pools'
 *                      layout with one byte per value), or [num_pages][kv_heads][page_size]
 *                      [head_dim] with pool.layout = KVC_HND
 *   k_scales, v_scales fp32 [num_pages][kv_heads][page_size] (the scales of one page and kv
 *                      head are contiguous)
 * All four 16-byte aligned; `pool` describes them as it describes a bf16 pool.
 *
 * kvc_store_int8 -- quantise and store new K/V at their slots (kvc_store's contract
 * otherwise: slot < 0 skipped, slots past the pool skipped and flagged).  Codes are
 * rint(x / scale) (ties to even) clamped to [-127, 127], with scale = max|x| / 127 and both
 * quotients computed in fp32 round-to-nearest; an all-zero vector stores scale 0 and codes 0.
 * Integer codes and scales are bit-exact.  k_new, v_new: bf16 [num_tokens][kv_heads][head_dim].
 */
kvc_status kvc_store_int8(void *k_codes, void *v_codes, float *k_scales, float *v_scales,
                          kvc_pool_desc pool, const void *k_new, const void *v_new,
                          const int32_t *slot_mapping, int32_t num_tokens, void *stream);

/*
 * kvc_decode_int8 -- kvc_decode over INT8 pages (same arguments and outputs).  Its work plan
 * differs from kvc_decode's split-K: for each kv head, the positions of all sequences (in
 * 64-position blocks, sequence after sequence) are cut into runs of equal cost (a block, plus
 * most of a block for each sequence a run starts), one CTA each, so that every CTA has the
 * same work however the context lengths are spread; a sequence covered by several runs has its
 * partial results merged (log-sum-exp) by a second launch.
 * kvc_decode_int8_plan gives the plan for num_splits: 0 = one wave of resident CTAs (the
 * default); 1 = one CTA per (sequence, kv head), no workspace and no merge; n > 1 = n runs
 * per sequence (num_seqs * n per kv head).  A plan never has more runs per kv head than
 * num_seqs * ceil(max_ctx / 64) (one per block), and at run time only as many runs as the
 * actual blocks are used.  splits_out = the number of CTAs, chunk_out = 64 (the block);
 * workspace_bytes_out = the workspace the call needs (0 for num_splits = 1).  head_dim 64 or
 * 128 (others: KVC_ERR_UNSUPPORTED).
 */
kvc_status kvc_decode_int8_plan(int32_t num_seqs, int32_t q_heads, kvc_pool_desc pool,
                                int32_t max_ctx, int32_t num_splits, int32_t *splits_out,
                                int32_t *chunk_out, size_t *workspace_bytes_out);
kvc_status kvc_decode_int8(void *out, int32_t out_dtype, const void *q, const void *k_codes,
                           const void *v_codes, const float *k_scales, const float *v_scales,
                           kvc_pool_desc pool, const int32_t *block_table, int32_t bt_stride,
                           const int32_t *context_lens, int32_t num_seqs, int32_t max_ctx,
                           int32_t q_heads, float scale, int32_t num_splits, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * kvc_decode_int8_store -- kvc_slot_mapping (one new token per sequence) + kvc_store_int8 +
 * kvc_decode_int8 in one call, as kvc_decode_store is for 16-bit pages (TileInfer.jl "KV
 * cache", "INT8 cache": a vector is quantised once, when it is written; "Pages and block
 * tables": the step writes the new key and value at their slot).  The decode CTA whose chunk
 * ends at sequence s's newest position (ctx_s - 1) quantises that token's key and value
 * (k_new[s], v_new[s], bf16 [num_seqs][kv_heads][128]) for its kv head with kvc_store_int8's
 * arithmetic, writes codes and scales at slot block_table[s][(ctx_s - 1) / page_size] *
 * page_size + (ctx_s - 1) % page_size before its own copies of that page, and the attention
 * reads them there.  Codes, scales and out end exactly as the three calls leave them.
 * Sequences with ctx_s = 0 store nothing; a slot past the pool is skipped and flagged
 * (kvc_device_errors).  Arguments as kvc_decode_int8 (split plan from kvc_decode_int8_plan),
 * plus k_new / v_new (device or pinned host memory, 16-byte aligned); the code and scale
 * pools are written.  out, q, block_table and context_lens may be pinned host memory, as for
 * kvc_decode.
 */
kvc_status kvc_decode_int8_store(void *out, int32_t out_dtype, const void *q, const void *k_new,
                                 const void *v_new, void *k_codes, void *v_codes,
                                 float *k_scales, float *v_scales, kvc_pool_desc pool,
                                 const int32_t *block_table, int32_t bt_stride,
                                 const int32_t *context_lens, int32_t num_seqs, int32_t max_ctx,
                                 int32_t q_heads, float scale, int32_t num_splits,
                                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * kvc_append_int8 -- kvc_append over INT8 pages (same arguments and outputs; the new tokens'
 * codes and scales must already be stored, kvc_store_int8).  The score of position p is
 * q . k_code[p] * k_scale[p] * scale and the value it weighs is v_scale[p] * v_code[p].  The
 * codes are exact operands of the tensor-core products (K as bf16 against the bf16 query, V
 * as fp16); the probability times the value scale enters the PV product as fp16 and the
 * softmax denominator sums the unrounded probabilities.  fp16's range limits value scales to
 * 4000 (|v| up to 5.08e5): a larger one sets a kvc_device_errors bit and its results are not
 * valid.  Positions past a sequence's context may hold any codes and NaN scales.  head_dim 64 or
 * 128 (others: KVC_ERR_UNSUPPORTED); NHD or HND pools.
 */
kvc_status kvc_append_int8(void *out, int32_t out_dtype, const void *q, const void *k_codes,
                           const void *v_codes, const float *k_scales, const float *v_scales,
                           kvc_pool_desc pool, const int32_t *block_table, int32_t bt_stride,
                           const int32_t *q_indptr, const int32_t *context_lens,
                           int32_t num_seqs, int32_t num_tokens, int32_t max_q_len,
                           int32_t max_ctx, int32_t q_heads, float scale, void *stream);

/*
 * kvc_copy_pages -- copy-on-write page copy ("KV Cache Management and PagedAttention", "Split
 * shared blocks when a write is needed": before a sequence writes into a page that other
 * sequences still reference, the page is copied to a new one and the writer's block-table
 * entry is pointed at the copy; Quail "KV", "Prefix sharing").  For every i < num_copies,
 * page dst_pages[i] of both pools receives the bytes of page src_pages[i] (all page_size
 * positions, all kv heads; a raw 16-bit copy, NaN payloads kept).  Deciding what to copy and
 * repointing the tables is host work (the caller's allocator and reference counts).
 *   src_pages, dst_pages  int32 [num_copies], device; ids in [0, num_pages)
 * Every copy reads the pools as they were before the call: a page that is both a source and a
 * destination in one call, or two copies to one destination, is a caller error (the result is
 * undefined).  Page ids outside the pool are skipped and set kvc_device_errors' range bit.
 */
kvc_status kvc_copy_pages(void *k_pool, void *v_pool, kvc_pool_desc pool,
                          const int32_t *src_pages, const int32_t *dst_pages,
                          int32_t num_copies, void *stream);

/*
 * kvc_validate -- opt-in deep check of the device-side tables of a step, for debugging
 * (no counterpart on the pages; every other call trusts these contents).  Checks, in order:
 *   1. 0 <= context_lens[s] <= bt_stride * page_size for every sequence s;
 *   2. every page id a sequence reaches, block_table[s][i] for i < ceil(context_lens[s] /
 *      page_size), lies in [0, num_pages)  (TileInfer.jl "KV cache", "Pages and block tables":
 *      a row lists the pages that hold the sequence's positions);
 *   3. every slot_mapping[t] is negative (padding, skipped by kvc_store) or below
 *      num_pages * page_size;
 *   4. no two tokens have the same non-negative slot (two writers of one slot in one store:
 *      "KV Cache Management and PagedAttention", "Split shared blocks when a write is needed",
 *      names that as the bug copy-on-write prevents).
 * block_table / context_lens may be NULL (num_seqs 0) to check slots only, and slot_mapping
 * NULL (num_tokens 0) to check tables only.  Unlike every other call it synchronises `stream`
 * and reads the verdict on the host.
 *   workspace      device bytes, at least *bytes_out of kvc_validate_workspace_size(pool)
 *                  (two bitmaps over the pool's slots and a verdict record); overwritten
 *   bad_index_out  host; on KVC_ERR_OUT_OF_RANGE the smallest offending index of the first
 *                  failing check (a sequence for checks 1-2, a token for 3-4; for 4 the
 *                  smallest token whose slot another token also writes), else -1
 * Returns KVC_OK when every check passes, KVC_ERR_OUT_OF_RANGE (kvc_last_error names the
 * check) when one fails, or an argument / CUDA error.
 */
kvc_status kvc_validate_workspace_size(kvc_pool_desc pool, size_t *bytes_out);
kvc_status kvc_validate(kvc_pool_desc pool, const int32_t *block_table, int32_t bt_stride,
                        const int32_t *context_lens, int32_t num_seqs,
                        const int32_t *slot_mapping, int32_t num_tokens, void *workspace,
                        size_t workspace_bytes, int64_t *bad_index_out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
