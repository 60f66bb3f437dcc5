// kvc_api.cu -- the C ABI declared in include/kvc.h: argument checks, split planning,
// TMA tensor-map encoding and kernel dispatch.  No device memory is allocated here.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdarg.h>
#include <algorithm>
#include <stdio.h>

#include <mutex>
#include <string>
#include <vector>

#include "kvc.h"
#include "kvc_launch.h"

namespace {

thread_local std::string g_last_error;
thread_local uint32_t *g_error_word = nullptr;   // kvc_set_error_word of this host thread

kvc_status fail(kvc_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

kvc_status ok()
{
    g_last_error.clear();
    return KVC_OK;
}

kvc_status cuda_fail(cudaError_t err, const char *what)
{
    return fail(KVC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(err));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kvc_status check_pool(const kvc_pool_desc &pool)
{
    if (pool.num_pages <= 0 || pool.page_size <= 0 || pool.kv_heads <= 0 || pool.head_dim <= 0)
        return fail(KVC_ERR_INVALID_ARG, "pool descriptor has a non-positive field");
    if (pool.head_dim != 64 && pool.head_dim != 128)
        return fail(KVC_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", pool.head_dim);
    if (pool.page_size != 16 && pool.page_size != 32 && pool.page_size != 64)
        return fail(KVC_ERR_UNSUPPORTED, "page_size %d (supported: 16, 32, 64)",
                    pool.page_size);
    if (static_cast<int64_t>(pool.num_pages) * pool.page_size >= (int64_t(1) << 31))
        return fail(KVC_ERR_UNSUPPORTED, "num_pages * page_size must be below 2^31");
    if (pool.layout != KVC_NHD && pool.layout != KVC_HND)
        return fail(KVC_ERR_INVALID_ARG, "layout %d (KVC_NHD or KVC_HND)", pool.layout);
    return KVC_OK;
}

kvc_status check_group(const kvc_pool_desc &pool, int32_t q_heads)
{
    if (q_heads <= 0 || q_heads % pool.kv_heads != 0)
        return fail(KVC_ERR_INVALID_ARG, "q_heads %d is not a multiple of kv_heads %d", q_heads,
                    pool.kv_heads);
    const int g = q_heads / pool.kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8)
        return fail(KVC_ERR_UNSUPPORTED, "GQA group %d (supported: 1, 2, 4, 8)", g);
    return KVC_OK;
}

int device_sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
        return n;
    cudaGetLastError();   // a host without a GPU: plan for a GB300
    return 152;
}

constexpr int kInt8Resident = 3;   // INT8 decode CTAs resident per SM (its automatic CTA count)

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
int64_t ceil_div(int64_t x, int64_t m) { return (x + m - 1) / m; }

struct Plan {
    int splits;
    int chunk;
    size_t ws_bytes;
    size_t lse_offset;
};

// Split-K plan.  Automatic splits aim at `ctas_per_sm_target` CTAs per SM over the whole
// launch: several waves of the kernel's resident CTAs, enough to spread the ramp and the
// uneven sequence lengths (bf16 decode: 2 resident CTAs per SM, target 4; INT8 decode: 3
// resident, target 12, measured best on the batched-decode workload).
Plan make_plan(int32_t num_seqs, int32_t q_heads, const kvc_pool_desc &pool, int32_t max_ctx,
               int32_t requested, int ctas_per_sm_target = 4)
{
    const int64_t ctx = max_ctx > 0 ? max_ctx : 1;
    const int64_t unit = kvc::kStageKeys;   // a multiple of every supported page size
    Plan p{};
    if (requested == 1) {
        p.splits = 1;
        p.chunk = static_cast<int>(round_up(ctx, unit));
    } else {
        int64_t want = requested;
        if (requested <= 0) {
            // Enough CTAs for several per SM: (sequence, kv head) units times splits.
            const int64_t units = static_cast<int64_t>(num_seqs > 0 ? num_seqs : 1) * pool.kv_heads;
            want = ceil_div(ctas_per_sm_target * static_cast<int64_t>(device_sm_count()),
                            units);
        }
        int64_t chunk = round_up(ceil_div(ctx, want), unit);
        if (requested <= 0 && chunk <= 2048 && ctas_per_sm_target < 8) {
            // Short chunks: the last CTAs to run set the tail and the merge is cheap, so the
            // positions are cut finer (measured on 64 sequences of U[512, 4096] positions: 3
            // splits 100.6 us against 2 splits 103.6; long contexts keep the coarser plan).
            const int64_t units =
                static_cast<int64_t>(num_seqs > 0 ? num_seqs : 1) * pool.kv_heads;
            want = ceil_div(8 * static_cast<int64_t>(device_sm_count()), units);
            chunk = round_up(ceil_div(ctx, want), unit);
        }
        if (requested <= 0 && chunk < 256)
            chunk = 256;
        p.chunk = static_cast<int>(chunk);
        p.splits = static_cast<int>(ceil_div(ctx, chunk));
    }
    if (p.splits > 1) {
        const size_t rows = static_cast<size_t>(num_seqs) * q_heads;
        const size_t o_bytes = rows * p.splits * pool.head_dim * sizeof(float);
        p.lse_offset = static_cast<size_t>(round_up(static_cast<int64_t>(o_bytes), 256));
        p.ws_bytes = p.lse_offset + rows * p.splits * sizeof(float);
    }
    return p;
}

// INT8 decode plan.  num_splits = 1: one CTA per (sequence, kv head) unit, no workspace.
// Otherwise each kv head's positions, in 64-position blocks over all sequences, are cut into
// `runs` runs of equal cost (the kernel weighs each sequence start against its blocks), one CTA
// per (run, kv head): one wave of resident CTAs (num_splits = 0) or
// num_splits runs per sequence, at most one per block.  Workspace: partial rows and
// log-sum-exps of kv_heads * (num_seqs + runs) slots, and (first slot, piece count) per unit.
struct Int8Plan {
    int ctas;
    bool per_unit;
    size_t ws_bytes, lse_offset, info_offset;
};

Int8Plan make_int8_plan(int32_t num_seqs, int32_t q_heads, const kvc_pool_desc &pool,
                        int32_t max_ctx, int32_t requested)
{
    Int8Plan p{};
    const int64_t seqs = num_seqs > 0 ? num_seqs : 1;
    const int64_t units = seqs * pool.kv_heads;
    if (requested == 1) {
        p.per_unit = true;
        p.ctas = static_cast<int>(units);
        return p;
    }
    const int64_t blocks = seqs * ceil_div(max_ctx > 0 ? max_ctx : 1, kvc::kStageKeys);
    int64_t runs = requested <= 0
                       ? kInt8Resident * static_cast<int64_t>(device_sm_count()) / pool.kv_heads
                       : static_cast<int64_t>(requested) * seqs;
    runs = std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(runs, blocks),
                                                  (int64_t(1) << 30) / pool.kv_heads));
    p.ctas = static_cast<int>(runs * pool.kv_heads);
    const int64_t group = q_heads / pool.kv_heads;
    const int64_t slots = pool.kv_heads * (seqs + runs);
    const int64_t o_bytes = slots * group * pool.head_dim * 4;
    p.lse_offset = static_cast<size_t>(round_up(o_bytes, 256));
    p.info_offset = static_cast<size_t>(
        round_up(static_cast<int64_t>(p.lse_offset) + slots * group * 4, 256));
    p.ws_bytes = p.info_offset + static_cast<size_t>(units) * 8;
    return p;
}

// ------------------------------------------------------------------------------------------
// TMA tensor maps over a pool viewed as [num_pages * page_size][kv_heads][head_dim] bf16,
// boxes of [page_size][1][64] with 128-byte swizzle.  Encoding is host work; the last few
// maps are memoised by (address, shape, device).
// ------------------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A tiled bf16 tensor map with 128-byte swizzle (boxes 64 elements wide), memoised by
// (address, shape, box, device).
struct MapKey {
    const void *ptr;
    int device;
    int rank;
    bool int8 = false;   // uint8 elements (INT8 pages) instead of bf16
    bool swizzle64 = false;   // 64-byte swizzle (rows of 64 bytes) instead of 128-byte
    cuuint64_t dims[4];
    cuuint64_t strides[3];
    cuuint32_t box[4];
    bool operator==(const MapKey &o) const
    {
        if (ptr != o.ptr || device != o.device || rank != o.rank || int8 != o.int8 ||
            swizzle64 != o.swizzle64)
            return false;
        for (int i = 0; i < rank; ++i)
            if (dims[i] != o.dims[i] || box[i] != o.box[i] ||
                (i + 1 < rank && strides[i] != o.strides[i]))
                return false;
        return true;
    }
};

struct MapEntry {
    MapKey key;
    CUtensorMap map;
};

std::mutex g_map_mutex;
std::vector<MapEntry> g_maps;   // most recent last, at most 32

kvc_status tensor_map(MapKey key, CUtensorMap *out)
{
    cudaError_t err = cudaGetDevice(&key.device);
    if (err != cudaSuccess)
        return cuda_fail(err, "cudaGetDevice");
    {
        std::lock_guard<std::mutex> lock(g_map_mutex);
        for (size_t i = g_maps.size(); i-- > 0;)
            if (g_maps[i].key == key) {
                *out = g_maps[i].map;
                return KVC_OK;
            }
    }
    auto fn = encode_fn();
    if (fn == nullptr)
        return fail(KVC_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint32_t elem_strides[4] = {1, 1, 1, 1};
    CUtensorMap map;
    CUresult r = fn(&map,
                    key.int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    static_cast<cuuint32_t>(key.rank),
                    const_cast<void *>(key.ptr), key.dims, key.strides, key.box, elem_strides,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    key.swizzle64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(KVC_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)",
                    static_cast<int>(r));
    std::lock_guard<std::mutex> lock(g_map_mutex);
    if (g_maps.size() >= 32)
        g_maps.erase(g_maps.begin());
    g_maps.push_back(MapEntry{key, map});
    *out = map;
    return KVC_OK;
}

// Pool [num_pages * page_size][kv_heads][head_dim] viewed as the 3-D tensor
// {head_dim, kv head, slot}; one box {64, 1, page_size} is one 64-column half of one page of
// one kv head (append: a 64-position stage is then [half][64 rows][64], one uniform operand).
kvc_status pool_tensor_map_halves(const void *base, const kvc_pool_desc &pool, CUtensorMap *out)
{
    MapKey k{};
    k.ptr = base;
    k.rank = 3;
    k.dims[0] = static_cast<cuuint64_t>(pool.head_dim);
    if (pool.layout == KVC_HND) {
        // {head_dim, offset, page * kv_heads + kv head}: box {64, page_size, 1}
        k.dims[1] = static_cast<cuuint64_t>(pool.page_size);
        k.dims[2] = static_cast<cuuint64_t>(pool.num_pages) * pool.kv_heads;
        k.strides[0] = static_cast<cuuint64_t>(pool.head_dim) * 2;
        k.strides[1] = static_cast<cuuint64_t>(pool.page_size) * pool.head_dim * 2;
        k.box[0] = 64;
        k.box[1] = static_cast<cuuint32_t>(pool.page_size);
        k.box[2] = 1;
        return tensor_map(k, out);
    }
    k.dims[1] = static_cast<cuuint64_t>(pool.kv_heads);
    k.dims[2] = static_cast<cuuint64_t>(pool.num_pages) * pool.page_size;
    k.strides[0] = static_cast<cuuint64_t>(pool.head_dim) * 2;
    k.strides[1] = static_cast<cuuint64_t>(pool.kv_heads) * pool.head_dim * 2;
    k.box[0] = 64;
    k.box[1] = 1;
    k.box[2] = static_cast<cuuint32_t>(pool.page_size);
    return tensor_map(k, out);
}

// New tokens' K or V [num_tokens][kv_heads][head_dim] bf16 viewed as {head_dim, kv head, token};
// one box {64, 1, page_size} is one column half of page_size consecutive tokens of one kv head,
// landing in shared memory exactly as a page box of an NHD pool does.
kvc_status new_tokens_tensor_map(const void *base, int32_t num_tokens, const kvc_pool_desc &pool,
                                 CUtensorMap *out)
{
    MapKey k{};
    k.ptr = base;
    k.rank = 3;
    k.dims[0] = static_cast<cuuint64_t>(pool.head_dim);
    k.dims[1] = static_cast<cuuint64_t>(pool.kv_heads);
    k.dims[2] = static_cast<cuuint64_t>(num_tokens);
    k.strides[0] = static_cast<cuuint64_t>(pool.head_dim) * 2;
    k.strides[1] = static_cast<cuuint64_t>(pool.kv_heads) * pool.head_dim * 2;
    k.box[0] = 64;
    k.box[1] = 1;
    k.box[2] = static_cast<cuuint32_t>(pool.page_size);
    return tensor_map(k, out);
}

// INT8 codes [num_pages * page_size][kv_heads][head_dim] viewed as the 3-D tensor
// {head_dim, kv head, slot} of bytes; one box {head_dim, 1, page_size} is one page of one kv
// head, [page_size rows][head_dim bytes] (128 bytes at head_dim 128, one swizzle row).  HND
// codes [num_pages][kv_heads][page_size][head_dim]: the tensor {head_dim, offset, page *
// kv_heads + kv head}, whose box {head_dim, page_size, 1} is the same contiguous block and
// lands in shared memory exactly as the NHD box does.
kvc_status pool_tensor_map_int8(const void *base, const kvc_pool_desc &pool, CUtensorMap *out)
{
    MapKey k{};
    k.ptr = base;
    k.rank = 3;
    k.int8 = true;
    k.swizzle64 = pool.head_dim == 64;   // 64-byte code rows: the 64-byte swizzle
    if (pool.layout == KVC_HND) {
        k.dims[0] = static_cast<cuuint64_t>(pool.head_dim);
        k.dims[1] = static_cast<cuuint64_t>(pool.page_size);
        k.dims[2] = static_cast<cuuint64_t>(pool.num_pages) * pool.kv_heads;
        k.strides[0] = static_cast<cuuint64_t>(pool.head_dim);
        k.strides[1] = static_cast<cuuint64_t>(pool.page_size) * pool.head_dim;
        k.box[0] = static_cast<cuuint32_t>(pool.head_dim);
        k.box[1] = static_cast<cuuint32_t>(pool.page_size);
        k.box[2] = 1;
        return tensor_map(k, out);
    }
    k.dims[0] = static_cast<cuuint64_t>(pool.head_dim);
    k.dims[1] = static_cast<cuuint64_t>(pool.kv_heads);
    k.dims[2] = static_cast<cuuint64_t>(pool.num_pages) * pool.page_size;
    k.strides[0] = static_cast<cuuint64_t>(pool.head_dim);
    k.strides[1] = static_cast<cuuint64_t>(pool.kv_heads) * pool.head_dim;
    k.box[0] = static_cast<cuuint32_t>(pool.head_dim);
    k.box[1] = 1;
    k.box[2] = static_cast<cuuint32_t>(pool.page_size);
    return tensor_map(k, out);
}

// Pool [num_pages * page_size][kv_heads][head_dim] viewed as the 4-D tensor
// {64 columns, slot, column half, kv head}; one box {64, page_size, head_dim / 64, 1} is a whole
// page of one kv head and lands in shared memory as [half][page_size rows][64 columns]
// (decode: one TMA instruction per page).
kvc_status pool_tensor_map(const void *base, const kvc_pool_desc &pool, CUtensorMap *out)
{
    MapKey k{};
    k.ptr = base;
    k.rank = 4;
    if (pool.layout == KVC_HND) {
        // {64 columns, offset, column half, page * kv_heads + kv head}: box {64, page_size,
        // head_dim / 64, 1} is one contiguous (page, kv head) block, [half][row][64] in smem
        k.dims[0] = 64;
        k.dims[1] = static_cast<cuuint64_t>(pool.page_size);
        k.dims[2] = static_cast<cuuint64_t>(pool.head_dim / 64);
        k.dims[3] = static_cast<cuuint64_t>(pool.num_pages) * pool.kv_heads;
        k.strides[0] = static_cast<cuuint64_t>(pool.head_dim) * 2;                   // row
        k.strides[1] = 128;                                                          // half
        k.strides[2] = static_cast<cuuint64_t>(pool.page_size) * pool.head_dim * 2;  // block
        k.box[0] = 64;
        k.box[1] = static_cast<cuuint32_t>(pool.page_size);
        k.box[2] = static_cast<cuuint32_t>(pool.head_dim / 64);
        k.box[3] = 1;
        return tensor_map(k, out);
    }
    k.dims[0] = 64;
    k.dims[1] = static_cast<cuuint64_t>(pool.num_pages) * pool.page_size;
    k.dims[2] = static_cast<cuuint64_t>(pool.head_dim / 64);
    k.dims[3] = static_cast<cuuint64_t>(pool.kv_heads);
    k.strides[0] = static_cast<cuuint64_t>(pool.kv_heads) * pool.head_dim * 2;   // slot
    k.strides[1] = 128;                                                           // half
    k.strides[2] = static_cast<cuuint64_t>(pool.head_dim) * 2;                    // kv head
    k.box[0] = 64;
    k.box[1] = static_cast<cuuint32_t>(pool.page_size);
    k.box[2] = static_cast<cuuint32_t>(pool.head_dim / 64);
    k.box[3] = 1;
    return tensor_map(k, out);
}

// Queries [T][q_heads][head_dim] viewed as [T][kv_heads][G][head_dim]; one box is the
// 128 / G tokens x G heads of one kv head (128 rows of 64 columns).
kvc_status query_tensor_map(const void *q, int32_t num_tokens, int32_t kv_heads, int32_t group,
                            int32_t head_dim, CUtensorMap *out)
{
    MapKey k{};
    k.ptr = q;
    k.rank = 4;
    k.dims[0] = static_cast<cuuint64_t>(head_dim);
    k.dims[1] = static_cast<cuuint64_t>(group);
    k.dims[2] = static_cast<cuuint64_t>(kv_heads);
    k.dims[3] = static_cast<cuuint64_t>(num_tokens);
    k.strides[0] = static_cast<cuuint64_t>(head_dim) * 2;
    k.strides[1] = static_cast<cuuint64_t>(group) * head_dim * 2;
    k.strides[2] = static_cast<cuuint64_t>(kv_heads) * group * head_dim * 2;
    k.box[0] = 64;
    k.box[1] = static_cast<cuuint32_t>(group);
    k.box[2] = 1;
    k.box[3] = static_cast<cuuint32_t>(128 / group);
    return tensor_map(k, out);
}

// Split plan of kvc_decode_shared_prefix: prefix chunks, then the suffix plan of kvc_decode.
struct GroupPlan {
    int prefix_chunk, n_prefix;
    Plan suffix;
    int stride;
    size_t lse_offset, key_start_offset, ws_bytes;
};

GroupPlan make_group_plan(int32_t num_seqs, int32_t q_heads, const kvc_pool_desc &pool,
                          int32_t max_ctx, int32_t num_groups, int32_t max_prefix_len)
{
    GroupPlan g{};
    const int64_t unit = kvc::kStageKeys;
    if (max_prefix_len > 0 && num_groups > 0) {
        const int64_t units = static_cast<int64_t>(num_groups) * pool.kv_heads;
        // as many prefix splits as keep the prefix CTAs within one wave of the grid's resident
        // CTAs (2 per SM), at least one: the rest of that wave takes suffix CTAs from the start
        // and no second wave of long prefix CTAs sets the tail (measured on 32 groups x 8
        // members with 2,048 shared positions, 256 (group, kv head) units: 1 split 102.9 us
        // against 105.0-107.0 for 2; 3, 4, 5 and 8 splits were slower still)
        const int64_t want =
            std::max<int64_t>(1, 2 * static_cast<int64_t>(device_sm_count()) / units);
        int64_t chunk = round_up(ceil_div(max_prefix_len, want), unit);
        if (chunk < 256)
            chunk = 256;
        g.prefix_chunk = static_cast<int>(chunk);
        g.n_prefix = static_cast<int>(ceil_div(max_prefix_len, chunk));
    }
    g.suffix = make_plan(num_seqs, q_heads, pool, max_ctx, 0);
    g.stride = g.n_prefix + g.suffix.splits;
    const size_t rows = static_cast<size_t>(num_seqs) * q_heads;
    const size_t o_bytes = rows * g.stride * pool.head_dim * sizeof(float);
    g.lse_offset = static_cast<size_t>(round_up(static_cast<int64_t>(o_bytes), 256));
    g.key_start_offset = static_cast<size_t>(
        round_up(static_cast<int64_t>(g.lse_offset + rows * g.stride * sizeof(float)), 256));
    g.ws_bytes = g.key_start_offset + static_cast<size_t>(num_seqs) * sizeof(int32_t);
    return g;
}

// Arguments that may live in host memory (the decode calls' out; the per-step inputs of slot
// mapping and store) must be device (or managed) memory, or pinned host memory that the
// device reaches at the same address (cudaHostAlloc / cudaHostRegister on a UVA system):
// kernels then read or write them across the host link directly.
kvc_status check_reachable(const void *p, const char *name)
{
    if (p == nullptr)
        return KVC_OK;   // optional, or nothing to do: checked by the caller
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return fail(KVC_ERR_INVALID_ARG, "%s: not a CUDA-visible pointer", name);
    }
    if (attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged)
        return KVC_OK;
    if (attr.type == cudaMemoryTypeHost && attr.devicePointer == p)
        return KVC_OK;
    return fail(KVC_ERR_INVALID_ARG,
                "%s must be device memory or pinned host memory mapped at its host address",
                name);
}

kvc_status check_decode_out(const void *out) { return check_reachable(out, "out"); }

kvc_status check_attention_args(const void *out, int32_t out_dtype, const void *q,
                                const void *k_pool, const void *v_pool,
                                const kvc_pool_desc &pool, const int32_t *block_table,
                                int32_t bt_stride, const int32_t *context_lens,
                                int32_t num_seqs, int32_t max_ctx, int32_t q_heads)
{
    kvc_status st = check_pool(pool);
    if (st != KVC_OK)
        return st;
    if ((st = check_group(pool, q_heads)) != KVC_OK)
        return st;
    if (out_dtype != KVC_BF16 && out_dtype != KVC_F32)
        return fail(KVC_ERR_INVALID_ARG, "out_dtype %d", out_dtype);
    if (num_seqs < 0 || num_seqs > 65535)
        return fail(KVC_ERR_INVALID_ARG, "num_seqs %d (0 .. 65535)", num_seqs);
    if (max_ctx < 0)
        return fail(KVC_ERR_INVALID_ARG, "max_ctx %d", max_ctx);
    if (bt_stride <= 0 || static_cast<int64_t>(bt_stride) * pool.page_size < max_ctx)
        return fail(KVC_ERR_INVALID_ARG, "bt_stride %d cannot hold max_ctx %d", bt_stride,
                    max_ctx);
    if (num_seqs > 0 && (!out || !q || !k_pool || !v_pool || !block_table || !context_lens))
        return fail(KVC_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return fail(KVC_ERR_INVALID_ARG, "q, out and pools must be 16-byte aligned");
    return KVC_OK;
}

}  // namespace

namespace kvc {
uint32_t *current_error_word()
{
    return g_error_word;
}
}  // namespace kvc

int kvc::set_last_error(int status, const char *message)
{
    g_last_error = message;
    return status;
}

extern "C" {

const char *kvc_status_string(kvc_status status)
{
    switch (status) {
    case KVC_OK: return "KVC_OK";
    case KVC_ERR_INVALID_ARG: return "KVC_ERR_INVALID_ARG";
    case KVC_ERR_UNSUPPORTED: return "KVC_ERR_UNSUPPORTED";
    case KVC_ERR_WORKSPACE: return "KVC_ERR_WORKSPACE";
    case KVC_ERR_CUDA: return "KVC_ERR_CUDA";
    case KVC_ERR_DEVICE: return "KVC_ERR_DEVICE";
    case KVC_ERR_OUT_OF_RANGE: return "KVC_ERR_OUT_OF_RANGE";
    }
    return "KVC_ERR_UNKNOWN";
}

const char *kvc_last_error(void) { return g_last_error.c_str(); }

kvc_status kvc_slot_mapping(int32_t *slot_mapping, const int32_t *block_table,
                            int32_t bt_stride, const int32_t *context_lens,
                            const int32_t *q_indptr, int32_t num_seqs, int32_t num_tokens,
                            int32_t max_q_len, int32_t page_size, void *stream)
{
    if (num_seqs < 0 || num_tokens < 0 || max_q_len < 0 || bt_stride <= 0 || page_size <= 0)
        return fail(KVC_ERR_INVALID_ARG, "negative size or non-positive stride/page size");
    if (q_indptr == nullptr && num_tokens != num_seqs)
        return fail(KVC_ERR_INVALID_ARG,
                    "without q_indptr every sequence has one token (num_tokens %d != %d)",
                    num_tokens, num_seqs);
    if (num_seqs > 0 && (!slot_mapping || !block_table || !context_lens))
        return fail(KVC_ERR_INVALID_ARG, "null pointer argument");
    if (num_seqs == 0 || num_tokens == 0)
        return ok();
    kvc_status st;
    if ((st = check_reachable(block_table, "block_table")) != KVC_OK ||
        (st = check_reachable(context_lens, "context_lens")) != KVC_OK ||
        (st = check_reachable(q_indptr, "q_indptr")) != KVC_OK)
        return st;
    cudaError_t err = kvc::launch_slot_mapping(slot_mapping, block_table, bt_stride,
                                               context_lens, q_indptr, num_seqs, num_tokens,
                                               max_q_len, page_size,
                                               static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? ok() : cuda_fail(err, "slot mapping launch");
}

kvc_status kvc_store(void *k_pool, void *v_pool, kvc_pool_desc pool, const void *k_new,
                     const void *v_new, const int32_t *slot_mapping, int32_t num_tokens,
                     void *stream)
{
    if (pool.num_pages <= 0 || pool.page_size <= 0 || pool.kv_heads <= 0 || pool.head_dim <= 0)
        return fail(KVC_ERR_INVALID_ARG, "pool descriptor has a non-positive field");
    if (num_tokens < 0)
        return fail(KVC_ERR_INVALID_ARG, "num_tokens %d", num_tokens);
    if ((static_cast<int64_t>(pool.kv_heads) * pool.head_dim * 2) % 16 != 0)
        return fail(KVC_ERR_UNSUPPORTED, "kv_heads * head_dim * 2 must be a multiple of 16");
    if (num_tokens == 0)
        return ok();
    if (!k_pool || !v_pool || !k_new || !v_new || !slot_mapping)
        return fail(KVC_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_new) || !aligned16(v_new))
        return fail(KVC_ERR_INVALID_ARG, "pools and new K/V must be 16-byte aligned");
    if (static_cast<int64_t>(pool.num_pages) * pool.page_size >= (int64_t(1) << 31))
        return fail(KVC_ERR_UNSUPPORTED, "num_pages * page_size must be below 2^31");
    if (pool.layout != KVC_NHD && pool.layout != KVC_HND)
        return fail(KVC_ERR_INVALID_ARG, "layout %d (KVC_NHD or KVC_HND)", pool.layout);
    kvc_status st;
    if ((st = check_reachable(k_new, "k_new")) != KVC_OK ||
        (st = check_reachable(v_new, "v_new")) != KVC_OK)
        return st;
    cudaError_t err = kvc::launch_store(k_pool, v_pool, pool.kv_heads, pool.head_dim,
                                        pool.num_pages * pool.page_size, k_new,
                                        v_new, slot_mapping, num_tokens,
                                        static_cast<cudaStream_t>(stream),
                                        pool.layout == KVC_HND, pool.page_size);
    return err == cudaSuccess ? ok() : cuda_fail(err, "store launch");
}

kvc_status kvc_decode_int8_plan(int32_t num_seqs, int32_t q_heads, kvc_pool_desc pool,
                                int32_t max_ctx, int32_t num_splits, int32_t *splits_out,
                                int32_t *chunk_out, size_t *workspace_bytes_out)
{
    kvc_status st = check_pool(pool);
    if (st != KVC_OK)
        return st;
    if (num_seqs < 0 || q_heads <= 0 || max_ctx < 0 || num_splits < 0)
        return fail(KVC_ERR_INVALID_ARG, "negative size or non-positive q_heads");
    if ((st = check_group(pool, q_heads)) != KVC_OK)
        return st;
    const Int8Plan p = make_int8_plan(num_seqs, q_heads, pool, max_ctx, num_splits);
    if (splits_out)
        *splits_out = p.ctas;
    if (chunk_out)
        *chunk_out = kvc::kStageKeys;
    if (workspace_bytes_out)
        *workspace_bytes_out = p.ws_bytes;
    return ok();
}

kvc_status kvc_store_int8(void *k_codes, void *v_codes, float *k_scales, float *v_scales,
                          kvc_pool_desc pool, const void *k_new, const void *v_new,
                          const int32_t *slot_mapping, int32_t num_tokens, void *stream)
{
    kvc_status st = check_pool(pool);
    if (st != KVC_OK)
        return st;
    if (num_tokens < 0)
        return fail(KVC_ERR_INVALID_ARG, "num_tokens %d", num_tokens);
    if (num_tokens == 0)
        return ok();
    if (!k_codes || !v_codes || !k_scales || !v_scales || !k_new || !v_new || !slot_mapping)
        return fail(KVC_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scales) ||
        !aligned16(v_scales) || !aligned16(k_new) || !aligned16(v_new))
        return fail(KVC_ERR_INVALID_ARG, "codes, scales and new K/V must be 16-byte aligned");
    cudaError_t err = kvc::launch_store_int8(k_codes, v_codes, k_scales, v_scales,
                                             pool.kv_heads, pool.head_dim, pool.page_size,
                                             pool.num_pages * pool.page_size, k_new, v_new,
                                             slot_mapping, num_tokens,
                                             static_cast<cudaStream_t>(stream),
                                             pool.layout == KVC_HND);
    return err == cudaSuccess ? ok() : cuda_fail(err, "store_int8 launch");
}

namespace {

// kvc_decode_int8, and kvc_decode_int8_store when k_new / v_new are given (the decode CTAs
// quantise and store the new tokens before reading their pages).
kvc_status decode_int8_impl(void *out, int32_t out_dtype, const void *q, const void *k_new,
                            const void *v_new, void *k_codes, void *v_codes, float *k_scales,
                            float *v_scales, kvc_pool_desc pool, const int32_t *block_table,
                            int32_t bt_stride, const int32_t *context_lens, int32_t num_seqs,
                            int32_t max_ctx, int32_t q_heads, float scale, int32_t num_splits,
                            void *workspace, size_t workspace_bytes, void *stream)
{
    kvc_status st = check_attention_args(out, out_dtype, q, k_codes, v_codes, pool, block_table,
                                         bt_stride, context_lens, num_seqs, max_ctx, q_heads);
    if (st != KVC_OK)
        return st;
    if (pool.head_dim != 64 && pool.head_dim != 128)
        return fail(KVC_ERR_UNSUPPORTED, "INT8 pages: head_dim %d (supported: 64, 128)",
                    pool.head_dim);
    if (!k_scales || !v_scales || !aligned16(k_scales) || !aligned16(v_scales))
        return fail(KVC_ERR_INVALID_ARG, "scales missing or not 16-byte aligned");
    if (num_splits < 0)
        return fail(KVC_ERR_INVALID_ARG, "num_splits %d", num_splits);
    if (num_seqs == 0)
        return ok();
    const Int8Plan p = make_int8_plan(num_seqs, q_heads, pool, max_ctx, num_splits);
    if (!p.per_unit) {
        if (workspace == nullptr || workspace_bytes < p.ws_bytes)
            return fail(KVC_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given",
                        p.ws_bytes, workspace == nullptr ? size_t(0) : workspace_bytes);
        if (!aligned16(workspace))
            return fail(KVC_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    }
    if ((st = check_decode_out(out)) != KVC_OK || (st = check_reachable(q, "q")) != KVC_OK ||
        (st = check_reachable(block_table, "block_table")) != KVC_OK ||
        (st = check_reachable(context_lens, "context_lens")) != KVC_OK)
        return st;
    const bool fused = k_new != nullptr || v_new != nullptr;
    if (fused) {
        if (!k_new || !v_new)
            return fail(KVC_ERR_INVALID_ARG, "null pointer argument");
        if (!aligned16(k_new) || !aligned16(v_new))
            return fail(KVC_ERR_INVALID_ARG, "new K/V must be 16-byte aligned");
        if (static_cast<int64_t>(pool.num_pages) * pool.page_size >= (int64_t(1) << 31))
            return fail(KVC_ERR_UNSUPPORTED, "num_pages * page_size must be below 2^31");
        if ((st = check_reachable(k_new, "k_new")) != KVC_OK ||
            (st = check_reachable(v_new, "v_new")) != KVC_OK)
            return st;
    }
    CUtensorMap tk, tv;
    if ((st = pool_tensor_map_int8(k_codes, pool, &tk)) != KVC_OK)
        return st;
    if ((st = pool_tensor_map_int8(v_codes, pool, &tv)) != KVC_OK)
        return st;
    kvc::DecodeInt8Launch l;
    l.q = q;
    l.k_scales = k_scales;
    l.v_scales = v_scales;
    l.out = out;
    l.out_f32 = out_dtype == KVC_F32;
    if (!p.per_unit) {
        l.part_o = static_cast<float *>(workspace);
        l.part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + p.lse_offset);
        l.unit_info = static_cast<char *>(workspace) + p.info_offset;
    }
    l.block_table = block_table;
    l.bt_stride = bt_stride;
    l.context_lens = context_lens;
    l.num_seqs = num_seqs;
    l.q_heads = q_heads;
    l.kv_heads = pool.kv_heads;
    l.page_size = pool.page_size;
    l.hnd = pool.layout == KVC_HND;
    l.head_dim = pool.head_dim;
    l.n_ctas = p.ctas;
    l.per_unit = p.per_unit;
    l.scale = scale > 0.0f ? scale : 1.0f / sqrtf(static_cast<float>(pool.head_dim));
    if (fused) {
        l.k_new = k_new;
        l.v_new = v_new;
        l.k_codes_w = k_codes;
        l.v_codes_w = v_codes;
        l.k_scales_w = k_scales;
        l.v_scales_w = v_scales;
        l.num_slots = pool.num_pages * pool.page_size;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t err = kvc::launch_decode_int8(l, tk, tv, s);
    if (err != cudaSuccess)
        return cuda_fail(err, "decode_int8 launch");
    return ok();
}

}  // namespace

kvc_status kvc_decode_int8(void *out, int32_t out_dtype, const void *q, const void *k_codes,
                           const void *v_codes, const float *k_scales, const float *v_scales,
                           kvc_pool_desc pool, const int32_t *block_table, int32_t bt_stride,
                           const int32_t *context_lens, int32_t num_seqs, int32_t max_ctx,
                           int32_t q_heads, float scale, int32_t num_splits, void *workspace,
                           size_t workspace_bytes, void *stream)
{
    return decode_int8_impl(out, out_dtype, q, nullptr, nullptr, const_cast<void *>(k_codes),
                            const_cast<void *>(v_codes), const_cast<float *>(k_scales),
                            const_cast<float *>(v_scales), pool, block_table, bt_stride,
                            context_lens, num_seqs, max_ctx, q_heads, scale, num_splits,
                            workspace, workspace_bytes, stream);
}

kvc_status kvc_decode_int8_store(void *out, int32_t out_dtype, const void *q, const void *k_new,
                                 const void *v_new, void *k_codes, void *v_codes,
                                 float *k_scales, float *v_scales, kvc_pool_desc pool,
                                 const int32_t *block_table, int32_t bt_stride,
                                 const int32_t *context_lens, int32_t num_seqs, int32_t max_ctx,
                                 int32_t q_heads, float scale, int32_t num_splits,
                                 void *workspace, size_t workspace_bytes, void *stream)
{
    if (num_seqs > 0 && (!k_new || !v_new))
        return fail(KVC_ERR_INVALID_ARG, "null pointer argument");
    return decode_int8_impl(out, out_dtype, q, k_new, v_new, k_codes, v_codes, k_scales,
                            v_scales, pool, block_table, bt_stride, context_lens, num_seqs,
                            max_ctx, q_heads, scale, num_splits, workspace, workspace_bytes,
                            stream);
}

kvc_status kvc_copy_pages(void *k_pool, void *v_pool, kvc_pool_desc pool,
                          const int32_t *src_pages, const int32_t *dst_pages,
                          int32_t num_copies, void *stream)
{
    if (pool.num_pages <= 0 || pool.page_size <= 0 || pool.kv_heads <= 0 || pool.head_dim <= 0)
        return fail(KVC_ERR_INVALID_ARG, "pool descriptor has a non-positive field");
    if (num_copies < 0)
        return fail(KVC_ERR_INVALID_ARG, "num_copies %d", num_copies);
    if ((static_cast<int64_t>(pool.page_size) * pool.kv_heads * pool.head_dim * 2) % 16 != 0)
        return fail(KVC_ERR_UNSUPPORTED, "a page must be a multiple of 16 bytes");
    if (num_copies == 0)
        return ok();
    if (!k_pool || !v_pool || !src_pages || !dst_pages)
        return fail(KVC_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned16(k_pool) || !aligned16(v_pool))
        return fail(KVC_ERR_INVALID_ARG, "pools must be 16-byte aligned");
    cudaError_t err = kvc::launch_copy_pages(k_pool, v_pool, pool.num_pages, pool.page_size,
                                             pool.kv_heads, pool.head_dim, src_pages, dst_pages,
                                             num_copies, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? ok() : cuda_fail(err, "copy_pages launch");
}

kvc_status kvc_decode_plan(int32_t num_seqs, int32_t q_heads, kvc_pool_desc pool,
                           int32_t max_ctx, int32_t num_splits, int32_t *splits_out,
                           int32_t *chunk_out, size_t *workspace_bytes_out)
{
    kvc_status st = check_pool(pool);
    if (st != KVC_OK)
        return st;
    if ((st = check_group(pool, q_heads)) != KVC_OK)
        return st;
    if (num_seqs < 0 || max_ctx < 0 || num_splits < 0)
        return fail(KVC_ERR_INVALID_ARG, "negative num_seqs, max_ctx or num_splits");
    const Plan p = make_plan(num_seqs, q_heads, pool, max_ctx, num_splits);
    if (splits_out)
        *splits_out = p.splits;
    if (chunk_out)
        *chunk_out = p.chunk;
    if (workspace_bytes_out)
        *workspace_bytes_out = p.ws_bytes;
    return ok();
}

}  // extern "C"

namespace {

// kvc_decode, and kvc_decode_store when k_new / v_new are given (the decode CTAs store the
// new tokens before reading their pages).
kvc_status decode_impl(void *out, int32_t out_dtype, const void *q, const void *k_new,
                       const void *v_new, void *k_pool, void *v_pool, kvc_pool_desc pool,
                       const int32_t *block_table, int32_t bt_stride,
                       const int32_t *context_lens, int32_t num_seqs, int32_t max_ctx,
                       int32_t q_heads, float scale, int32_t num_splits, void *workspace,
                       size_t workspace_bytes, void *stream)
{
    kvc_status st = check_attention_args(out, out_dtype, q, k_pool, v_pool, pool, block_table,
                                         bt_stride, context_lens, num_seqs, max_ctx, q_heads);
    if (st != KVC_OK)
        return st;
    if (num_splits < 0)
        return fail(KVC_ERR_INVALID_ARG, "num_splits %d", num_splits);
    if (num_seqs == 0)
        return ok();
    const Plan p = make_plan(num_seqs, q_heads, pool, max_ctx, num_splits);
    if (p.splits > 1) {
        if (workspace == nullptr || workspace_bytes < p.ws_bytes)
            return fail(KVC_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given",
                        p.ws_bytes, workspace == nullptr ? size_t(0) : workspace_bytes);
        if (!aligned16(workspace))
            return fail(KVC_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    }
    if ((st = check_decode_out(out)) != KVC_OK || (st = check_reachable(q, "q")) != KVC_OK ||
        (st = check_reachable(block_table, "block_table")) != KVC_OK ||
        (st = check_reachable(context_lens, "context_lens")) != KVC_OK)
        return st;
    const bool fused = k_new != nullptr || v_new != nullptr;
    if (fused) {
        if (!k_new || !v_new)
            return fail(KVC_ERR_INVALID_ARG, "null pointer argument");
        if (!aligned16(k_new) || !aligned16(v_new))
            return fail(KVC_ERR_INVALID_ARG, "new K/V must be 16-byte aligned");
        if (static_cast<int64_t>(pool.num_pages) * pool.page_size >= (int64_t(1) << 31))
            return fail(KVC_ERR_UNSUPPORTED, "num_pages * page_size must be below 2^31");
        if ((st = check_reachable(k_new, "k_new")) != KVC_OK ||
            (st = check_reachable(v_new, "v_new")) != KVC_OK)
            return st;
    }
    CUtensorMap tk, tv;
    if ((st = pool_tensor_map(k_pool, pool, &tk)) != KVC_OK)
        return st;
    if ((st = pool_tensor_map(v_pool, pool, &tv)) != KVC_OK)
        return st;
    kvc::DecodeLaunch l;
    l.q = q;
    l.out = out;
    l.out_f32 = out_dtype == KVC_F32;
    l.part_o = static_cast<float *>(workspace);
    l.part_lse = p.splits > 1 ? reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                                          p.lse_offset)
                              : nullptr;
    l.block_table = block_table;
    l.bt_stride = bt_stride;
    l.context_lens = context_lens;
    l.num_seqs = num_seqs;
    l.q_heads = q_heads;
    l.kv_heads = pool.kv_heads;
    l.head_dim = pool.head_dim;
    l.page_size = pool.page_size;
    l.chunk = p.chunk;
    l.n_split = p.splits;
    l.scale = scale > 0.0f ? scale : 1.0f / sqrtf(static_cast<float>(pool.head_dim));
    l.hnd = pool.layout == KVC_HND;
    if (fused) {
        l.k_new = k_new;
        l.v_new = v_new;
        l.k_pool_w = k_pool;
        l.v_pool_w = v_pool;
        l.num_slots = pool.num_pages * pool.page_size;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t err = kvc::launch_decode(l, tk, tv, s);
    if (err != cudaSuccess)
        return cuda_fail(err, "decode launch");
    if (p.splits > 1) {
        err = kvc::launch_merge(out, l.out_f32, l.part_o, l.part_lse, num_seqs * q_heads,
                                p.splits, pool.head_dim, nullptr, s);
        if (err != cudaSuccess)
            return cuda_fail(err, "merge launch");
    }
    return ok();
}

}  // namespace

extern "C" {

kvc_status kvc_decode(void *out, int32_t out_dtype, const void *q, const void *k_pool,
                      const void *v_pool, kvc_pool_desc pool, const int32_t *block_table,
                      int32_t bt_stride, const int32_t *context_lens, int32_t num_seqs,
                      int32_t max_ctx, int32_t q_heads, float scale, int32_t num_splits,
                      void *workspace, size_t workspace_bytes, void *stream)
{
    return decode_impl(out, out_dtype, q, nullptr, nullptr, const_cast<void *>(k_pool),
                       const_cast<void *>(v_pool), pool, block_table, bt_stride, context_lens,
                       num_seqs, max_ctx, q_heads, scale, num_splits, workspace,
                       workspace_bytes, stream);
}

kvc_status kvc_decode_store(void *out, int32_t out_dtype, const void *q, const void *k_new,
                            const void *v_new, void *k_pool, void *v_pool, kvc_pool_desc pool,
                            const int32_t *block_table, int32_t bt_stride,
                            const int32_t *context_lens, int32_t num_seqs, int32_t max_ctx,
                            int32_t q_heads, float scale, int32_t num_splits, void *workspace,
                            size_t workspace_bytes, void *stream)
{
    if (num_seqs > 0 && (!k_new || !v_new))
        return fail(KVC_ERR_INVALID_ARG, "null pointer argument");
    return decode_impl(out, out_dtype, q, k_new, v_new, k_pool, v_pool, pool, block_table,
                       bt_stride, context_lens, num_seqs, max_ctx, q_heads, scale, num_splits,
                       workspace, workspace_bytes, stream);
}

kvc_status kvc_shared_prefix_groups(const int32_t *block_table, int32_t bt_stride,
                                    const int32_t *context_lens, int32_t num_seqs,
                                    int32_t page_size, int32_t max_members,
                                    int32_t *group_indptr, int32_t *group_seqs,
                                    int32_t *prefix_len, int32_t *num_groups, void *stream)
{
    if (num_seqs < 0 || num_seqs > 65535)
        return fail(KVC_ERR_INVALID_ARG, "num_seqs %d (0 .. 65535)", num_seqs);
    if (page_size <= 0 || bt_stride <= 0)
        return fail(KVC_ERR_INVALID_ARG, "page_size %d, bt_stride %d", page_size, bt_stride);
    if (max_members < 2 || max_members > 64)
        return fail(KVC_ERR_INVALID_ARG, "max_members %d (2 .. 64)", max_members);
    if (!group_indptr || !num_groups || (num_seqs > 0 && (!block_table || !context_lens ||
                                                          !group_seqs)) ||
        (num_seqs > 1 && !prefix_len))
        return fail(KVC_ERR_INVALID_ARG, "null pointer argument");
    const cudaError_t err = kvc::launch_group_detect(
        block_table, bt_stride, context_lens, num_seqs, page_size, max_members, group_indptr,
        group_seqs, prefix_len, num_groups, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? ok() : cuda_fail(err, "group detection launch");
}

kvc_status kvc_decode_shared_prefix_plan(int32_t num_seqs, int32_t q_heads, kvc_pool_desc pool,
                                         int32_t max_ctx, int32_t num_groups,
                                         int32_t max_prefix_len, size_t *workspace_bytes_out)
{
    kvc_status st = check_pool(pool);
    if (st != KVC_OK)
        return st;
    if ((st = check_group(pool, q_heads)) != KVC_OK)
        return st;
    if (num_seqs < 0 || max_ctx < 0 || num_groups < 0 || max_prefix_len < 0)
        return fail(KVC_ERR_INVALID_ARG, "negative size");
    const GroupPlan g = make_group_plan(num_seqs, q_heads, pool, max_ctx, num_groups,
                                        max_prefix_len);
    if (workspace_bytes_out)
        *workspace_bytes_out = g.ws_bytes;
    return ok();
}

kvc_status kvc_decode_shared_prefix(void *out, int32_t out_dtype, const void *q,
                                    const void *k_pool, const void *v_pool, kvc_pool_desc pool,
                                    const int32_t *block_table, int32_t bt_stride,
                                    const int32_t *context_lens, int32_t num_seqs,
                                    int32_t max_ctx, int32_t q_heads, float scale,
                                    const int32_t *group_indptr, const int32_t *group_seqs,
                                    const int32_t *prefix_len, int32_t num_groups,
                                    int32_t max_group_size, int32_t max_prefix_len,
                                    void *workspace, size_t workspace_bytes, void *stream)
{
    kvc_status st = check_attention_args(out, out_dtype, q, k_pool, v_pool, pool, block_table,
                                         bt_stride, context_lens, num_seqs, max_ctx, q_heads);
    if (st != KVC_OK)
        return st;
    if (num_groups < 0 || max_group_size < 0 || max_prefix_len < 0 || max_prefix_len > max_ctx)
        return fail(KVC_ERR_INVALID_ARG, "bad group sizes (0 <= max_prefix_len <= max_ctx)");
    const int G = q_heads / pool.kv_heads;
    if (static_cast<int64_t>(max_group_size) * G > 64)
        return fail(KVC_ERR_UNSUPPORTED,
                    "a group's query rows (members x q_heads / kv_heads = %d) exceed 64",
                    max_group_size * G);
    if (num_groups > 65535)
        return fail(KVC_ERR_INVALID_ARG, "num_groups %d (at most 65535)", num_groups);
    if (num_groups > 0 && (!group_indptr || !group_seqs || !prefix_len))
        return fail(KVC_ERR_INVALID_ARG, "null group array");
    if (num_seqs == 0)
        return ok();
    const GroupPlan g = make_group_plan(num_seqs, q_heads, pool, max_ctx, num_groups,
                                        max_prefix_len);
    if (workspace == nullptr || workspace_bytes < g.ws_bytes)
        return fail(KVC_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", g.ws_bytes,
                    workspace == nullptr ? size_t(0) : workspace_bytes);
    if (!aligned16(workspace))
        return fail(KVC_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    CUtensorMap tk, tv;
    if ((st = pool_tensor_map(k_pool, pool, &tk)) != KVC_OK)
        return st;
    if ((st = pool_tensor_map(v_pool, pool, &tv)) != KVC_OK)
        return st;
    char *ws = static_cast<char *>(workspace);
    float *part_o = reinterpret_cast<float *>(ws);
    float *part_lse = reinterpret_cast<float *>(ws + g.lse_offset);
    int32_t *key_start = reinterpret_cast<int32_t *>(ws + g.key_start_offset);
    const float sc = scale > 0.0f ? scale : 1.0f / sqrtf(static_cast<float>(pool.head_dim));
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    cudaError_t err = kvc::launch_grouped_setup(key_start, group_indptr, group_seqs, prefix_len,
                                                num_groups, num_seqs, pool.page_size, bt_stride,
                                                s);
    if (err != cudaSuccess)
        return cuda_fail(err, "grouped setup launch");
    kvc::GroupedPrefixLaunch p;
    p.q = q;
    p.part_o = part_o;
    p.part_lse = part_lse;
    p.block_table = block_table;
    p.bt_stride = bt_stride;
    p.group_indptr = group_indptr;
    p.group_seqs = group_seqs;
    p.prefix_len = prefix_len;
    p.num_groups = num_groups;
    p.max_rows = max_group_size * G;
    p.num_seqs = num_seqs;
    p.q_heads = q_heads;
    p.kv_heads = pool.kv_heads;
    p.head_dim = pool.head_dim;
    p.page_size = pool.page_size;
    p.chunk = g.prefix_chunk;
    p.n_split = g.n_prefix;
    p.split_stride = g.stride;
    p.scale = sc;
    p.hnd = pool.layout == KVC_HND;
    kvc::DecodeLaunch l;
    l.q = q;
    l.out = out;
    l.out_f32 = out_dtype == KVC_F32;
    l.part_o = part_o;
    l.part_lse = part_lse;
    l.block_table = block_table;
    l.bt_stride = bt_stride;
    l.context_lens = context_lens;
    l.num_seqs = num_seqs;
    l.q_heads = q_heads;
    l.kv_heads = pool.kv_heads;
    l.head_dim = pool.head_dim;
    l.page_size = pool.page_size;
    l.chunk = g.suffix.chunk;
    l.n_split = g.suffix.splits;
    l.scale = sc;
    l.key_start = key_start;
    l.split_base = g.n_prefix;
    l.split_stride = g.stride;
    l.hnd = pool.layout == KVC_HND;
    // one resident wave (2 per SM) of prefix CTAs at most: the empty slots of a group list
    // found on the device then cost one load each instead of a CTA start
    p.max_prefix_ctas = 2 * device_sm_count();
    if (g.n_prefix == 0)
        p.num_groups = 0;   // no prefix CTAs
    if ((err = kvc::launch_grouped_decode(p, l, tk, tv, s)) != cudaSuccess)
        return cuda_fail(err, "grouped prefix + suffix decode launch");
    if ((err = kvc::launch_merge(out, l.out_f32, part_o, part_lse, num_seqs * q_heads, g.stride,
                                 pool.head_dim, nullptr, s)) != cudaSuccess)
        return cuda_fail(err, "merge launch");
    return ok();
}

kvc_status kvc_merge(void *out, int32_t out_dtype, const float *partial_o,
                     const float *partial_lse, int32_t rows, int32_t num_splits,
                     int32_t head_dim, float *lse_out, void *stream)
{
    if (out_dtype != KVC_BF16 && out_dtype != KVC_F32)
        return fail(KVC_ERR_INVALID_ARG, "out_dtype %d", out_dtype);
    if (rows < 0 || num_splits <= 0)
        return fail(KVC_ERR_INVALID_ARG, "rows %d, num_splits %d", rows, num_splits);
    if (head_dim != 64 && head_dim != 128)
        return fail(KVC_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
    if (rows == 0)
        return ok();
    if (!out || !partial_o || !partial_lse)
        return fail(KVC_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned16(partial_o) || !aligned16(out))
        return fail(KVC_ERR_INVALID_ARG, "partial_o and out must be 16-byte aligned");
    if (kvc_status st = check_decode_out(out); st != KVC_OK)
        return st;
    cudaError_t err = kvc::launch_merge(out, out_dtype == KVC_F32, partial_o, partial_lse, rows,
                                        num_splits, head_dim, lse_out,
                                        static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? ok() : cuda_fail(err, "merge launch");
}

kvc_status kvc_append(void *out, int32_t out_dtype, const void *q, const void *k_pool,
                      const void *v_pool, kvc_pool_desc pool, const int32_t *block_table,
                      int32_t bt_stride, const int32_t *q_indptr,
                      const int32_t *context_lens, int32_t num_seqs, int32_t num_tokens,
                      int32_t max_q_len, int32_t max_ctx, int32_t q_heads, float scale,
                      void *stream)
{
    kvc_status st = check_attention_args(out, out_dtype, q, k_pool, v_pool, pool, block_table,
                                         bt_stride, context_lens, num_seqs, max_ctx, q_heads);
    if (st != KVC_OK)
        return st;
    if (num_tokens < 0 || max_q_len < 0)
        return fail(KVC_ERR_INVALID_ARG, "num_tokens %d, max_q_len %d", num_tokens, max_q_len);
    if (num_seqs > 0 && q_indptr == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "q_indptr is required");
    if (static_cast<int64_t>(max_q_len) * (q_heads / pool.kv_heads) > (int64_t(1) << 30))
        return fail(KVC_ERR_INVALID_ARG, "max_q_len too large");
    if (num_seqs == 0 || num_tokens == 0 || max_q_len == 0)
        return ok();
    CUtensorMap tq, tk, tv;
    if ((st = pool_tensor_map_halves(k_pool, pool, &tk)) != KVC_OK)
        return st;
    if ((st = pool_tensor_map_halves(v_pool, pool, &tv)) != KVC_OK)
        return st;
    if ((st = query_tensor_map(q, num_tokens, pool.kv_heads, q_heads / pool.kv_heads,
                               pool.head_dim, &tq)) != KVC_OK)
        return st;
    kvc::AppendLaunch l;
    l.q = q;
    l.out = out;
    l.out_f32 = out_dtype == KVC_F32;
    l.block_table = block_table;
    l.bt_stride = bt_stride;
    l.q_indptr = q_indptr;
    l.context_lens = context_lens;
    l.num_seqs = num_seqs;
    l.num_tokens = num_tokens;
    l.max_q_len = max_q_len;
    l.q_heads = q_heads;
    l.kv_heads = pool.kv_heads;
    l.head_dim = pool.head_dim;
    l.page_size = pool.page_size;
    l.scale = scale > 0.0f ? scale : 1.0f / sqrtf(static_cast<float>(pool.head_dim));
    l.hnd = pool.layout == KVC_HND;
    cudaError_t err = kvc::launch_append_tc(l, tq, tk, tv, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? ok() : cuda_fail(err, "append launch");
}

kvc_status kvc_append_store(void *out, int32_t out_dtype, const void *q, const void *k_new,
                            const void *v_new, void *k_pool, void *v_pool, kvc_pool_desc pool,
                            const int32_t *block_table, int32_t bt_stride,
                            const int32_t *q_indptr, const int32_t *context_lens,
                            int32_t num_seqs, int32_t num_tokens, int32_t max_q_len,
                            int32_t max_ctx, int32_t q_heads, float scale, void *stream)
{
    kvc_status st = check_attention_args(out, out_dtype, q, k_pool, v_pool, pool, block_table,
                                         bt_stride, context_lens, num_seqs, max_ctx, q_heads);
    if (st != KVC_OK)
        return st;
    if (num_tokens < 0 || max_q_len < 0)
        return fail(KVC_ERR_INVALID_ARG, "num_tokens %d, max_q_len %d", num_tokens, max_q_len);
    if (num_seqs > 0 && q_indptr == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "q_indptr is required");
    if (num_tokens > 0 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)))
        return fail(KVC_ERR_INVALID_ARG, "k_new / v_new missing or not 16-byte aligned");
    if (static_cast<int64_t>(max_q_len) * (q_heads / pool.kv_heads) > (int64_t(1) << 30))
        return fail(KVC_ERR_INVALID_ARG, "max_q_len too large");
    if (num_seqs == 0 || num_tokens == 0 || max_q_len == 0)
        return ok();
    CUtensorMap tq, tk, tv, tkn, tvn;
    if ((st = pool_tensor_map_halves(k_pool, pool, &tk)) != KVC_OK)
        return st;
    if ((st = pool_tensor_map_halves(v_pool, pool, &tv)) != KVC_OK)
        return st;
    // Plan: with pages of 64 positions or more, the chunk's first page (stored before the
    // append, since cached positions share it) holds most of a short chunk, and the fused
    // append's gain (the rest of the chunk read once) no longer pays for its ring slots living
    // until their rows are written: the whole chunk is stored first and the plain append
    // follows (measured on the rewind workload: fused 2% faster at P 16, 2% slower at P 64).
    const bool whole = pool.page_size >= 64;
    if (!whole) {
        if ((st = new_tokens_tensor_map(k_new, num_tokens, pool, &tkn)) != KVC_OK)
            return st;
        if ((st = new_tokens_tensor_map(v_new, num_tokens, pool, &tvn)) != KVC_OK)
            return st;
    }
    if ((st = query_tensor_map(q, num_tokens, pool.kv_heads, q_heads / pool.kv_heads,
                               pool.head_dim, &tq)) != KVC_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t err = kvc::launch_store_boundary(
        k_pool, v_pool, pool.kv_heads, pool.head_dim, pool.page_size,
        pool.num_pages * pool.page_size, pool.layout == KVC_HND, k_new, v_new, block_table,
        bt_stride, q_indptr, context_lens, num_seqs, whole, s);
    if (err != cudaSuccess)
        return cuda_fail(err, "boundary store launch");
    kvc::AppendLaunch l;
    l.q = q;
    l.out = out;
    l.out_f32 = out_dtype == KVC_F32;
    l.block_table = block_table;
    l.bt_stride = bt_stride;
    l.q_indptr = q_indptr;
    l.context_lens = context_lens;
    l.num_seqs = num_seqs;
    l.num_tokens = num_tokens;
    l.max_q_len = max_q_len;
    l.q_heads = q_heads;
    l.kv_heads = pool.kv_heads;
    l.head_dim = pool.head_dim;
    l.page_size = pool.page_size;
    l.scale = scale > 0.0f ? scale : 1.0f / sqrtf(static_cast<float>(pool.head_dim));
    l.hnd = pool.layout == KVC_HND;
    if (whole) {
        err = kvc::launch_append_tc(l, tq, tk, tv, s);
    } else {
        l.fused = true;
        l.k_pool_w = k_pool;
        l.v_pool_w = v_pool;
        l.num_pages = pool.num_pages;
        err = kvc::launch_append_tc(l, tq, tk, tv, s, &tkn, &tvn);
    }
    return err == cudaSuccess ? ok() : cuda_fail(err, "append launch");
}

kvc_status kvc_append_int8(void *out, int32_t out_dtype, const void *q, const void *k_codes,
                           const void *v_codes, const float *k_scales, const float *v_scales,
                           kvc_pool_desc pool, const int32_t *block_table, int32_t bt_stride,
                           const int32_t *q_indptr, const int32_t *context_lens,
                           int32_t num_seqs, int32_t num_tokens, int32_t max_q_len,
                           int32_t max_ctx, int32_t q_heads, float scale, void *stream)
{
    kvc_status st = check_attention_args(out, out_dtype, q, k_codes, v_codes, pool, block_table,
                                         bt_stride, context_lens, num_seqs, max_ctx, q_heads);
    if (st != KVC_OK)
        return st;
    if (pool.head_dim != 64 && pool.head_dim != 128)
        return fail(KVC_ERR_UNSUPPORTED, "INT8 pages: head_dim %d (supported: 64, 128)",
                    pool.head_dim);
    if (!k_scales || !v_scales || !aligned16(k_scales) || !aligned16(v_scales))
        return fail(KVC_ERR_INVALID_ARG, "scales missing or not 16-byte aligned");
    if (num_tokens < 0 || max_q_len < 0)
        return fail(KVC_ERR_INVALID_ARG, "num_tokens %d, max_q_len %d", num_tokens, max_q_len);
    if (num_seqs > 0 && q_indptr == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "q_indptr is required");
    if (static_cast<int64_t>(max_q_len) * (q_heads / pool.kv_heads) > (int64_t(1) << 30))
        return fail(KVC_ERR_INVALID_ARG, "max_q_len too large");
    if (num_seqs == 0 || num_tokens == 0 || max_q_len == 0)
        return ok();
    CUtensorMap tq, tk, tv;
    if ((st = pool_tensor_map_int8(k_codes, pool, &tk)) != KVC_OK)
        return st;
    if ((st = pool_tensor_map_int8(v_codes, pool, &tv)) != KVC_OK)
        return st;
    if ((st = query_tensor_map(q, num_tokens, pool.kv_heads, q_heads / pool.kv_heads,
                               pool.head_dim, &tq)) != KVC_OK)
        return st;
    kvc::AppendInt8Launch l;
    l.out = out;
    l.out_f32 = out_dtype == KVC_F32;
    l.k_scales = k_scales;
    l.v_scales = v_scales;
    l.block_table = block_table;
    l.bt_stride = bt_stride;
    l.q_indptr = q_indptr;
    l.context_lens = context_lens;
    l.num_seqs = num_seqs;
    l.num_tokens = num_tokens;
    l.max_q_len = max_q_len;
    l.q_heads = q_heads;
    l.kv_heads = pool.kv_heads;
    l.page_size = pool.page_size;
    l.head_dim = pool.head_dim;
    l.hnd = pool.layout == KVC_HND;
    l.scale = scale > 0.0f ? scale : 1.0f / sqrtf(static_cast<float>(pool.head_dim));
    cudaError_t err = kvc::launch_append_int8(l, tq, tk, tv, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? ok() : cuda_fail(err, "append_int8 launch");
}

kvc_status kvc_set_error_word(uint32_t *device_word)
{
    if ((reinterpret_cast<uintptr_t>(device_word) & 3u) != 0)
        return fail(KVC_ERR_INVALID_ARG, "error word not 4-byte aligned");
    g_error_word = device_word;
    return ok();
}

kvc_status kvc_selftest_wait(void *stream)
{
    const cudaError_t err = kvc::launch_selftest_wait(static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? ok() : cuda_fail(err, "self-test launch");
}

kvc_status kvc_device_errors(uint32_t *flags_out)
{
    if (flags_out == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "flags_out is null");
    uint32_t a = 0, c = 0, d = 0;
    cudaError_t err = kvc::read_and_clear_decode_errors(&a);
    if (err == cudaSuccess)
        err = kvc::read_and_clear_store_errors(&c);
    uint32_t e = 0;
    if (err == cudaSuccess)
        err = kvc::read_and_clear_append_tc_errors(&d);
    if (err == cudaSuccess)
        err = kvc::read_and_clear_grouped_errors(&e);
    uint32_t f = 0;
    if (err == cudaSuccess)
        err = kvc::read_and_clear_decode_int8_errors(&f);
    e |= f;
    if (err == cudaSuccess)
        err = kvc::read_and_clear_append_int8_errors(&f);
    e |= f;
    if (err != cudaSuccess)
        return cuda_fail(err, "reading the device error word");
    *flags_out = a | c | d | e;
    return *flags_out ? fail(KVC_ERR_DEVICE, "device error flags 0x%x", *flags_out) : ok();
}

kvc_status kvc_validate_workspace_size(kvc_pool_desc pool, size_t *bytes_out)
{
    if (bytes_out == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "bytes_out is null");
    kvc_status st = check_pool(pool);
    if (st != KVC_OK)
        return st;
    *bytes_out = kvc::validate_workspace_bytes(static_cast<long long>(pool.num_pages) *
                                               pool.page_size);
    return ok();
}

kvc_status kvc_validate(kvc_pool_desc pool, const int32_t *block_table, int32_t bt_stride,
                        const int32_t *context_lens, int32_t num_seqs,
                        const int32_t *slot_mapping, int32_t num_tokens, void *workspace,
                        size_t workspace_bytes, int64_t *bad_index_out, void *stream)
{
    if (bad_index_out == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "bad_index_out is null");
    *bad_index_out = -1;
    kvc_status st = check_pool(pool);
    if (st != KVC_OK)
        return st;
    if (num_seqs < 0 || num_tokens < 0)
        return fail(KVC_ERR_INVALID_ARG, "negative num_seqs %d or num_tokens %d", num_seqs,
                    num_tokens);
    if (num_seqs > 0 && (block_table == nullptr || context_lens == nullptr || bt_stride <= 0))
        return fail(KVC_ERR_INVALID_ARG, "tables missing or bt_stride %d", bt_stride);
    if (num_tokens > 0 && slot_mapping == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "slot_mapping is null");
    const size_t need =
        kvc::validate_workspace_bytes(static_cast<long long>(pool.num_pages) * pool.page_size);
    if (workspace == nullptr || workspace_bytes < need ||
        (reinterpret_cast<uintptr_t>(workspace) & 3u) != 0)
        return fail(KVC_ERR_WORKSPACE, "workspace of %zu bytes (4-byte aligned) needed", need);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t err = kvc::launch_validate(block_table, bt_stride, context_lens, num_seqs,
                                           slot_mapping, num_tokens, pool.page_size,
                                           pool.num_pages, workspace, s);
    kvc::ValidateRecord rec;
    if (err == cudaSuccess)
        err = cudaMemcpyAsync(&rec, workspace, sizeof(rec), cudaMemcpyDeviceToHost, s);
    if (err == cudaSuccess)
        err = cudaStreamSynchronize(s);
    if (err != cudaSuccess)
        return cuda_fail(err, "validate");
    static const char *const kWhat[kvc::kValidateChecks] = {
        "context_lens[s] outside [0, bt_stride * page_size]",
        "page id outside [0, num_pages)",
        "slot past the pool",
        "slot written by two tokens"};
    for (int c = 0; c < kvc::kValidateChecks; ++c)
        if (rec.first_bad[c] != 0x7FFFFFFF) {
            *bad_index_out = rec.first_bad[c];
            return fail(KVC_ERR_OUT_OF_RANGE, "%s (index %d)", kWhat[c], rec.first_bad[c]);
        }
    return ok();
}

}  // extern "C"
