// tc_common.cuh -- tensor-core (tcgen05), tensor-memory, mbarrier and TMA
// helpers shared by the prefill kernels (sm_100 family, inline PTX).
//
// Shared-memory operand tiles are 128-byte-swizzled panels of 64 16-bit
// elements: 16-byte chunk c of row r of a panel sits at (c ^ (r mod 8)) * 16
// within the row's 128 bytes, the layout a SWIZZLE_128B TMA box lands in and
// the K-major (or, read the other way, MN-major) layout the tensor core reads.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pkv_common.cuh"

namespace pkv {
namespace tc {

constexpr uint32_t kSpin = 1u << 22;   // try_wait rounds before a wait gives up

__device__ __forceinline__ uint32_t s_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Offset of 16-byte chunk `c` (along the row) of row `r` in a tile of `rows`
// rows stored as 128-byte-swizzled panels of 64 16-bit elements.
__device__ __forceinline__ uint32_t panel_off(int r, int c, int rows)
{
    return (uint32_t)((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Instruction descriptor of kind::f16 with an fp32 accumulator.
template <int CT>
__device__ __forceinline__ uint32_t instr_desc(int m, int n, int b_mn_major)
{
    const uint32_t ab = CT == kBF16 ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)b_mn_major << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// D (tensor memory) (+)= A (shared memory) B (shared memory), kind::f16, one
// CTA.  The shared-memory matrix descriptors come as 32-bit halves (see
// desc_lo / desc_hi), so that a loop over K steps only adds to the low halves.
__device__ __forceinline__ void umma_h(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi,
                                       uint32_t b_lo, uint32_t b_hi, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile("{\n .reg .pred p;\n .reg .b64 da, db;\n setp.ne.b32 p, %6, 0;\n"
                 " mov.b64 da, {%1, %2};\n mov.b64 db, {%3, %4};\n"
                 " tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n}" ::"r"(d_tmem),
                 "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate));
}

// D (tensor memory) (+)= A (tensor memory) B (shared memory), the same way.
__device__ __forceinline__ void umma_ts_h(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                          uint32_t b_hi, uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n .reg .pred p;\n .reg .b64 db;\n setp.ne.b32 p, %5, 0;\n"
                 " mov.b64 db, {%2, %3};\n"
                 " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n}" ::"r"(d_tmem),
                 "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate));
}

// Shared-memory matrix descriptor of the sm_100 family, 128-byte swizzle, as
// two 32-bit halves.  Low: start address >> 4 (bits 0-13), leading-dimension
// byte offset >> 4 (bits 16-29).  High: stride-dimension byte offset >> 4
// (bits 0-13), descriptor version 1 (bit 14), swizzle mode 2 = 128-byte
// (bits 29-31).
__host__ __device__ constexpr uint32_t desc_lo(uint32_t addr, uint32_t lbo)
{
    return ((addr >> 4) & 0x3fffu) | (((lbo >> 4) & 0x3fffu) << 16);
}
__host__ __device__ constexpr uint32_t desc_hi(uint32_t sbo)
{
    return ((sbo >> 4) & 0x3fffu) | (1u << 14) | (2u << 29);
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same test without suspending: one look at the phase.
__device__ __forceinline__ bool test_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of parity `parity` of `bar`; false after kSpin polls or
// kWaitNs nanoseconds.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity)
{
    WaitClock clock;
    for (uint32_t i = 0; i < kSpin; ++i)
        if (try_wait(bar, parity))
            return true;
        else if (clock.expired(i))
            break;
    return false;
}

__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void bar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Add `bytes` to the transaction count without arriving.
__device__ __forceinline__ void bar_expect_only(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// generic-proxy shared-memory writes -> visible to the async proxy (TMA, tensor core)
__device__ __forceinline__ void async_proxy_fence() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 16 consecutive 32-bit columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                 "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
                 "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                     taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                 "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// TMA: one box {64 elements, BS rows} of a 2-D tensor map into shared memory,
// completing transaction bytes on an mbarrier.
__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap* map, int x, int y,
                                        uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// tma_box with an L2 cache policy for the lines it reads
__device__ __forceinline__ void tma_box_hint(uint32_t dst, const CUtensorMap* map, int x, int y,
                                             uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// 16 bytes global -> shared, or 16 zero bytes when !valid
__device__ __forceinline__ void cp16z(uint32_t dst, const void* src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two floats -> two 16-bit elements (first in the low half), round to nearest even.
template <int CT>
__device__ __forceinline__ uint32_t pack_rn(float a, float b)
{
    uint32_t r;
    if constexpr (CT == kBF16)
        asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(a), "f"(b));
    else
        asm("cvt.rn.f16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(a), "f"(b));
    return r;
}

// Two fp32 lanes per instruction (sm_100 family): a b + c, a + b, a - b.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    float2 r;
    asm("{\n .reg .b64 ra, rb, rc, rd;\n"
        " mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
        " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b)
{
    float2 r;
    asm("{\n .reg .b64 ra, rb, rd;\n"
        " mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
        " add.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

__device__ __forceinline__ float2 fsub2(float2 a, float2 b)
{
    float2 r;
    asm("{\n .reg .b64 ra, rb, rd;\n"
        " mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
        " sub.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

// max of three (a NaN operand is ignored, as fmaxf does)
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime.
inline EncodeTiled encoder()
{
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(f);
    });
    return fn;
}

// The cache as a 2-D tensor [num_blocks * num_kv_heads * BS rows][D] of 16-bit
// elements; boxes of 64 elements x BS rows land 128-byte swizzled, rows
// outside the tensor as zeros.
inline bool cache_map(CUtensorMap* map, const void* cache, int64_t rows, int D, int BS)
{
    EncodeTiled enc = encoder();
    if (enc == nullptr || rows <= 0 || rows >= (int64_t)1 << 31)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)BS};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(cache), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc
}  // namespace pkv
