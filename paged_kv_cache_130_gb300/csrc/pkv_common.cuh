// pkv_common.cuh -- element types, vector memory access and conversions shared
// by the paged KV-cache kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

constexpr int kF16 = PKV_F16;
constexpr int kBF16 = PKV_BF16;
constexpr int kE4M3 = PKV_FP8_E4M3;

constexpr float kLog2e = 1.4426950408889634f;

template <int DT>
struct Elem {
    static constexpr int bytes = (DT == kE4M3) ? 1 : 2;
    static constexpr int per_vec = 16 / bytes;     // elements in one 16-byte vector
};

// ------------------------------------------------------------------ loads

// An L2 policy for data read once (K/V tiles, for the bulk and tensor copies
// that take a cache hint): its lines are the first to go when L2 needs room,
// so that a stream of them does not push out other lines (such as those an
// earlier kernel wrote and L2 has not yet written back).
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 16-byte load of data that is read once (K/V tiles): skip L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void* p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 16-byte read-only load through the normal cached path.
__device__ __forceinline__ uint4 ld_ro(const void* p)
{
    return __ldg(reinterpret_cast<const uint4*>(p));
}

// 16-byte shared-memory read.
__device__ __forceinline__ uint4 ld_shared16(const void* p)
{
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
    return r;
}

// 16-byte global -> shared asynchronous copy (L2 only), grouped per thread
// with commit / wait_group: the wait covers this thread's own copies.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
                 "l"(gsrc)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void st_v4(void* p, uint4 v)
{
    *reinterpret_cast<uint4*>(p) = v;
}

// ------------------------------------------------------------------ conversions

// Two packed 16-bit values (low half = element 0) to float.
template <int DT>
__device__ __forceinline__ float2 unpack2(uint32_t w);

template <>
__device__ __forceinline__ float2 unpack2<kF16>(uint32_t w)
{
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
}

template <>
__device__ __forceinline__ float2 unpack2<kBF16>(uint32_t w)
{
    // bfloat16 is the upper half of an fp32 value
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Four E4M3 codes (byte i = element i) -> two f16 pairs (elements 0, 1 and
// 2, 3), each exact; the conversions read the word's 16-bit halves directly.
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi)
{
    asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n"
        " cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t h)
{
    __half2 hh = *reinterpret_cast<__half2*>(&h);
    return __half22float2(hh);
}

// 16 bytes of cache data -> EPV floats.
template <int DT>
__device__ __forceinline__ void unpack_vec(const uint4& v, float* out)
{
    if constexpr (DT == kE4M3) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t lo, hi;
            e4m3x4_to_f16x2(w[i], lo, hi);
            const float2 a = f16x2_to_float2(lo);
            const float2 b = f16x2_to_float2(hi);
            out[4 * i + 0] = a.x;
            out[4 * i + 1] = a.y;
            out[4 * i + 2] = b.x;
            out[4 * i + 3] = b.y;
        }
    } else {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 a = unpack2<DT>(w[i]);
            out[2 * i + 0] = a.x;
            out[2 * i + 1] = a.y;
        }
    }
}

// fp32 -> 16-bit element bits, round to nearest even.
template <int DT>
__device__ __forceinline__ uint16_t round_to(float x)
{
    if constexpr (DT == kF16) {
        return __half_as_ushort(__float2half_rn(x));
    } else {
        return __bfloat16_as_ushort(__float2bfloat16_rn(x));
    }
}

__device__ __forceinline__ uint32_t pack2(uint16_t lo, uint16_t hi)
{
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// Two floats -> two E4M3 codes (low byte = first), round to nearest even,
// saturating to the largest finite value.
__device__ __forceinline__ uint16_t e4m3x2_satfinite(float a, float b)
{
    return static_cast<uint16_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// ------------------------------------------------------------------ misc

// Every mbarrier wait in these kernels is bounded in polls and in time: a
// try_wait poll may suspend the thread for a while of the hardware's choosing,
// so a limit on polls alone does not bound how long a wait for a phase that
// never completes takes.  A wait also gives up kWaitNs nanoseconds (by
// %globaltimer) after its first failed poll.
constexpr uint64_t kWaitNs = 1000000000ull;

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// The time bound of one wait; expired(i) after failed poll i (from 0).
struct WaitClock {
    uint64_t t0 = 0;
    __device__ __forceinline__ bool expired(uint32_t i)
    {
        const uint64_t now = global_ns();
        if (i == 0) {
            t0 = now;
            return false;
        }
        return now - t0 > kWaitNs;
    }
};

__device__ __forceinline__ void flag_error(int32_t* dev_err, int32_t bit)
{
    if (dev_err != nullptr)
        atomicOr(dev_err, bit);
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue; wait until the previous kernel's memory is visible.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait_primary()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace pkv
