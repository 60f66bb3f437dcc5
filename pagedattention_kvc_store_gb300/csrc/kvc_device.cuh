// kvc_device.cuh -- device-side building blocks shared by the kvc kernels (sm_103a).
//
// Inline PTX for: mbarriers with bounded waits, TMA tensor loads (cp.async.bulk.tensor),
// ldmatrix, and the bf16 m16n8k16 tensor-core MMA used where the tile is thin.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
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
    kErrAppendTcWait = 1u << 8,    // the tcgen05 append gave up a wait
    kErrSmemAlign = 1u << 9,       // dynamic shared memory not 1024-byte aligned: no work done
    kErrPageRange = 1u << 10,      // a page copy named a page outside the pool: skipped
    kErrScaleRange = 1u << 11,     // INT8 append: a value scale above its fp16 limit (4000)
    kErrSelftestWait = 1u << 12,   // kvc_selftest_wait: its wait ran out, as it must
};

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch.  Every kvc kernel starts with pdl_wait() -- it returns once
// the grids this launch depends on have completed and their writes are visible (at once when
// the launch has no such dependency) -- and then pdl_trigger(), which lets the next launch on
// the stream start its CTAs as this grid's last ones are scheduled; they wait in their own
// pdl_wait().  The next kernel's launch and prologue so overlap this one's tail.
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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

// Non-blocking: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
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

// Untiled bulk copy global -> shared, completion counted on an mbarrier (both addresses
// 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes),
        "r"(smem_addr(bar))
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

// c[16x8] += a[16x16] * b[16x8] with fp16 operands (fp32 accumulate).
__device__ __forceinline__ void mma_f16_16816(float (&c)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------------------
// tcgen05: tensor memory (TMEM) and the 5th-generation tensor-core MMA
// ---------------------------------------------------------------------------------------

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile.  K-major tiles:
// rows of 128 bytes, 8-row groups `sbo` bytes apart (lbo unused).  MN-major tiles: 64
// contiguous MN elements per 128-byte row, K rows 128 bytes apart, 8-row K groups `sbo`
// apart and 64-element MN groups `lbo` apart.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_byte_addr, uint32_t lbo,
                                                    uint32_t sbo)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_byte_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;   // descriptor version for tcgen05
    d |= 2ull << 61;   // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, M x N, K-major A; B K-major
// (b_mn = 0) or MN-major (b_mn = 1).
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, int b_mn)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(b_mn) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// The same with fp16 A and B (type field 0).
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N, int b_mn)
{
    return (1u << 4) | (static_cast<uint32_t>(b_mn) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]; issued by one thread.
__device__ __forceinline__ void umma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]; A is M lanes x K columns of tensor memory, column j of a
// 16-bit A holding elements 2j (low half) and 2j + 1 (high half) of the row.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane from raw words (warp-collective).
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane from raw words (warp-collective).
__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t *slot_in_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(slot_in_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async proxy
// (TMA, tensor cores).
// A 16-byte read-only load that does not allocate in L1 (data read once).
__device__ __forceinline__ uint4 load_streaming(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Orders this thread's earlier generic-proxy global accesses before its later async-proxy
// (TMA) ones.
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 4-D tiled tensor load with an L2 cache-policy hint (used for K/V pages).
__device__ __forceinline__ void tma_load_4d_hint(void *dst, const CUtensorMap *map, int c0, int c1,
                                                 int c2, int c3, uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// 4-D tiled tensor load (used for query tiles).
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, int c3, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(smem_addr(bar))
        : "memory");
}

// 2^x with the hardware approximation (ex2.approx, ~2 ulp); 2^-inf = +0.
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Paired fp32 arithmetic of the sm_100 family: two fp32 lanes in one 64-bit register, one
// instruction for both (round-to-nearest, like the scalar operations).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// max(a, b, c) in one instruction (sm_100 family).
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Two 16x16 matrices of bytes from shared memory, transposed (ldmatrix .m16n16 .trans .b8):
// lanes 0-15 give the 16-byte rows of matrix 0, lanes 16-31 those of matrix 1.  Lane l
// (g = l / 4, t = l % 4) receives, per matrix, the bytes of rows 4t .. 4t + 3 in column g (d0)
// and in column g + 8 (d1).  Ordered after earlier volatile asm (the mbarrier waits).
__device__ __forceinline__ void ldsm_x2_trans_b8(uint32_t addr, uint32_t &d0, uint32_t &d1,
                                                 uint32_t &d2, uint32_t &d3)
{
    asm volatile("ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0, %1, %2, %3}, [%4];"
                 : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
                 : "r"(addr));
}

// Transpose of an 8x8 matrix of 16-bit values held as one register per lane (lane l: row
// l / 4, columns 2 (l % 4) and 2 (l % 4) + 1): lane l receives row l / 4 of the transpose.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x)
{
    uint32_t y;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Both fp16 pairs of one word of int8 codes (codes 0, 1 and codes 2, 3), exact: the word's
// sign bits flipped (m = code + 128), the bytes put under exponent 0x64 and 1152 subtracted.
__device__ __forceinline__ void codes_word_f16x2(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    const uint32_t m = w ^ 0x80808080u;
    const uint32_t e = 0x64646464u;
    const uint32_t a = __byte_perm(m, e, 0x4140u);   // [m.0, 0x64, m.1, 0x64]
    const uint32_t b = __byte_perm(m, e, 0x4342u);   // [m.2, 0x64, m.3, 0x64]
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2 *>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
    lo = *reinterpret_cast<const uint32_t *>(&ha);
    hi = *reinterpret_cast<const uint32_t *>(&hb);
}

// Both bf16 pairs of one word of int8 codes (codes 0, 1 and codes 2, 3), exact.  A code's low
// seven bits m go under the exponent of 128 (bf16 128 + m: the step is 1 on [128, 256)); the
// code is then 128 + m minus 128, or minus 256 where its sign bit is set (two's complement).
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ void codes_word_bf16x2(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    const uint32_t e = 0x43434343u;
    const uint32_t a = __byte_perm(w, e, 0x4140u);   // [c.0, 0x43, c.1, 0x43]
    const uint32_t b = __byte_perm(w, e, 0x4342u);   // [c.2, 0x43, c.3, 0x43]
    lo = bf16x2_sub(a & 0xFF7FFF7Fu, (a & 0x00800080u) | 0x43004300u);
    hi = bf16x2_sub(b & 0xFF7FFF7Fu, (b & 0x00800080u) | 0x43004300u);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// One output element, fp32 or bf16 (round to nearest even) as the caller's out_f32 says.
__device__ __forceinline__ void store_out(void *out, int out_f32, size_t idx, float v)
{
    if (out_f32)
        static_cast<float *>(out)[idx] = v;
    else
        static_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
}

// Two consecutive outputs from element idx (even): one 8- or 4-byte store.
__device__ __forceinline__ void store_out2(void *out, int out_f32, size_t idx, float2 v)
{
    if (out_f32)
        *reinterpret_cast<float2 *>(static_cast<float *>(out) + idx) = v;
    else
        *reinterpret_cast<uint32_t *>(static_cast<__nv_bfloat16 *>(out) + idx) =
            pack_bf16x2(v.x, v.y);
}

// Four consecutive outputs from element idx (a multiple of 4): one 16- or 8-byte store.
__device__ __forceinline__ void store_out4(void *out, int out_f32, size_t idx, float4 v)
{
    if (out_f32) {
        *reinterpret_cast<float4 *>(static_cast<float *>(out) + idx) = v;
    } else {
        uint2 packed;
        packed.x = pack_bf16x2(v.x, v.y);
        packed.y = pack_bf16x2(v.z, v.w);
        *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(out) + idx) = packed;
    }
}

// Sum of the two bf16 values packed in v (exact widening to fp32).  Softmax sums are taken
// over the rounded probabilities that the PV product actually uses, so that numerator and
// denominator weigh every position the same.
__device__ __forceinline__ float bf16x2_sum(uint32_t v)
{
    return __uint_as_float(v << 16) + __uint_as_float(v & 0xFFFF0000u);
}

// Keep the bf16 halves of `v` whose key index is below `n_valid`; zero the others.
__device__ __forceinline__ uint32_t keep_keys(uint32_t v, int key_lo, int n_valid)
{
    uint32_t lo = (key_lo < n_valid) ? 0x0000FFFFu : 0u;
    uint32_t hi = (key_lo + 1 < n_valid) ? 0xFFFF0000u : 0u;
    return v & (lo | hi);
}

// Byte offset, inside a stage tile of whole pages, of the 16-byte chunk holding element
// column `col` (bf16 index in 0..head_dim-1) of row `row` (position in the stage).  Each page
// of `page_rows` rows is stored [half][page_rows][64] bf16 (128 bytes per row) by one TMA box
// with 128-byte swizzling: inside each 1024-byte block of 8 rows, chunk c of row r sits at
// chunk c ^ (r & 7).  page_rows is a multiple of 8.
template <int D>
__device__ __forceinline__ uint32_t page_tile_offset(int row, int col, int log2_page_rows)
{
    const int page = row >> log2_page_rows;
    const int r = row & ((1 << log2_page_rows) - 1);
    const int half = col >> 6;
    const int chunk = (col & 63) >> 3;
    return static_cast<uint32_t>((page * (D / 64) + half) << (log2_page_rows + 7)) +
           static_cast<uint32_t>(r * 128 + ((chunk ^ (r & 7)) << 4));
}

}  // namespace kvc
