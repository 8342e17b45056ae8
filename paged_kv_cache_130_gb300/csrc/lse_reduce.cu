// lse_reduce.cu -- merge of split-context partitions (log-sum-exp reduce).
//
// For every (sequence, query head) whose context spans two or more
// partitions: M = max_p m_p, w_p = 2^(m_p - M),
// out = sum_p w_p o_p / sum_p w_p l_p.  One CTA per (s, h), one thread per
// output dim; the per-partition weights go through shared memory.  Launched
// with programmatic dependent launch: the prologue (index math, context
// length) overlaps the partition kernel's tail, and griddepcontrol.wait orders
// the partial reads after that kernel's writes.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kReduceThreads = 128;
constexpr int kMaxCachedParts = 512;      // weights kept in shared memory

template <int QT>
__global__ void __launch_bounds__(kReduceThreads) lse_reduce_kernel(const ReduceParams p)
{
    __shared__ float sm_w[kMaxCachedParts];
    __shared__ float sm_red[kReduceThreads / 32];
    __shared__ float sm_inv_l;

    const int row = blockIdx.x;                       // s * num_heads + h
    const int s = row / p.num_heads;
    const int ctx = __ldg(p.context_lens + s);
    if (ctx < 0 || ctx > p.max_context_len)
        return;
    const int npart = (ctx + p.partition_size - 1) / p.partition_size;
    if (npart <= 1)
        return;

    pdl_wait_primary();

    const int64_t base = (int64_t)row * p.max_partitions;
    const float* m = p.ws_m + base;
    const float* l = p.ws_l + base;

    // M = max_p m_p
    float mx = -CUDART_INF_F;
    for (int i = threadIdx.x; i < npart; i += blockDim.x)
        mx = fmaxf(mx, m[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if ((threadIdx.x & 31) == 0)
        sm_red[threadIdx.x >> 5] = mx;
    __syncthreads();
    float M = sm_red[0];
#pragma unroll
    for (int i = 1; i < kReduceThreads / 32; ++i)
        M = fmaxf(M, sm_red[i]);
    __syncthreads();

    // weights and their l-weighted sum
    float lsum = 0.f;
    for (int i = threadIdx.x; i < npart; i += blockDim.x) {
        const float wi = (M == -CUDART_INF_F || m[i] == -CUDART_INF_F) ? 0.f : exp2f(m[i] - M);
        if (i < kMaxCachedParts)
            sm_w[i] = wi;
        lsum += wi * l[i];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    if ((threadIdx.x & 31) == 0)
        sm_red[threadIdx.x >> 5] = lsum;
    __syncthreads();
    if (threadIdx.x == 0) {
        float L = 0.f;
#pragma unroll
        for (int i = 0; i < kReduceThreads / 32; ++i)
            L += sm_red[i];
        sm_inv_l = L > 0.f ? 1.f / L : 0.f;
    }
    __syncthreads();
    const float inv_l = sm_inv_l;

    const int D = p.head_dim;
    uint16_t* out = reinterpret_cast<uint16_t*>(p.out) + (int64_t)row * D;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        const float* o = p.ws_o + base * D + d;
        float acc = 0.f;
        for (int i = 0; i < npart; ++i) {
            const float wi = i < kMaxCachedParts
                                 ? sm_w[i]
                                 : ((M == -CUDART_INF_F || m[i] == -CUDART_INF_F)
                                        ? 0.f : exp2f(m[i] - M));
            if (wi != 0.f)
                acc = fmaf(wi, o[(int64_t)i * D], acc);
        }
        out[d] = round_to<QT>(acc * inv_l);
    }
}

}  // namespace

cudaError_t launch_lse_reduce(const ReduceParams& p, cudaStream_t stream, bool pdl)
{
    const int64_t rows = (int64_t)p.num_seqs * p.num_heads;
    if (rows <= 0 || p.max_partitions <= 1)
        return cudaSuccess;
    if (rows > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows);
    cfg.blockDim = dim3(kReduceThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (p.out_dtype == kF16)
        return cudaLaunchKernelEx(&cfg, lse_reduce_kernel<kF16>, p);
    if (p.out_dtype == kBF16)
        return cudaLaunchKernelEx(&cfg, lse_reduce_kernel<kBF16>, p);
    return cudaErrorNotSupported;
}

}  // namespace pkv
