// kvc_device.cuh -- device-side building blocks shared by the kvc kernels (sm_103a).
//
// Inline PTX for: mbarriers with bounded waits, TMA tensor loads (cp.async.bulk.tensor),
// ldmatrix, and the bf16 m16n8k16 tensor-core MMA used where the tile is thin.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kvc {

// A bounded wait gives up after about this many SM cycles (~1 s at GB300 clocks).
constexpr long long kWaitLimitCycles = 2000000000LL;

// Bits of the device error word (kvc_device_errors).
enum DeviceErrorBits : uint32_t {
    kErrDecodeFullWait = 1u << 0,
    kErrDecodeEmptyWait = 1u << 1,
    kErrAppendFullWait = 1u << 2,
    kErrAppendEmptyWait = 1u << 3,
    kErrAppendMmaWait = 1u << 4,
    kErrDrainWait = 1u << 5,
    kErrSlotRange = 1u << 6,       // a store slot past the pool: the token was skipped
    kErrContextRange = 1u << 7,    // context_lens[s] > bt_stride * page_size: clamped
};

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait until the phase with the given parity has completed.  Returns false (and the caller
// must give up) if that takes longer than kWaitLimitCycles.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long start = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - start > kWaitLimitCycles)
            return false;
    }
    return true;
}

// Named barrier over `count` threads (a multiple of 32), id 1..15.
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------------------------------
// TMA: 3-D tiled tensor load into shared memory, completion counted on an mbarrier.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar)),
        "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    return policy;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(policy));
    return policy;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------------------
// ldmatrix / mma.sync (bf16 in, fp32 accumulate)
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                              uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// c[16x8] += a[16x16] * b[16x8]; a row-major fragments a0..a3, b column fragments b0, b1.
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^x with the hardware approximation (ex2.approx, ~2 ulp); 2^-inf = +0.
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Keep the bf16 halves of `v` whose key index is below `n_valid`; zero the others.
__device__ __forceinline__ uint32_t keep_keys(uint32_t v, int key_lo, int n_valid)
{
    uint32_t lo = (key_lo < n_valid) ? 0x0000FFFFu : 0u;
    uint32_t hi = (key_lo + 1 < n_valid) ? 0xFFFF0000u : 0u;
    return v & (lo | hi);
}

// Byte offset, inside a stage tile written by TMA with 128-byte swizzling, of the 16-byte
// chunk holding element column `col` (bf16 index in 0..head_dim-1) of row `row`.  The tile
// is stored as head_dim/64 column halves of [rows][64] bf16 (128 bytes per row); inside a
// 1024-byte block of 8 rows, chunk c of row r sits at chunk c ^ (r & 7).
template <int ROWS>
__device__ __forceinline__ uint32_t swz_offset(int row, int col)
{
    const int half = col >> 6;
    const int chunk = (col & 63) >> 3;
    return static_cast<uint32_t>(half * ROWS * 128 + row * 128 + ((chunk ^ (row & 7)) << 4));
}

}  // namespace kvc
