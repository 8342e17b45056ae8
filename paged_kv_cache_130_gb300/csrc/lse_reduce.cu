// lse_reduce.cu -- merge of split-context partitions (log-sum-exp reduce).
//
// For every (sequence, query head) whose context spans two or more
// partitions, or that has a shared prefix: M = max_p m_p, w_p = 2^(m_p - M),
// out = sum_p w_p o_p / sum_p w_p l_p.  With a shared prefix of P tokens the
// partials are the ceil(P / prefix_partition) partitions of the prefix
// followed by those of the rest of the context.
// One warp per (sequence, head) row: lanes read the row's m and l strided,
// reduce M and the weighted l with shuffles, then every lane accumulates its
// D/32 output dims over the partitions, many vector loads in flight at once.
// Launched with programmatic dependent launch: the context length is read
// before griddepcontrol.wait (it is an input, not a partial), the partials
// after it.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "decode_common.cuh"
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kRowsPerCta = 4;
constexpr int kFewParts = 8;           // rows with this many partials or fewer: one load round

template <int QT, int D>
__global__ void __launch_bounds__(kRowsPerCta * 32) lse_reduce_kernel(const ReduceParams p)
{
    constexpr int DPL = D / 32;                       // dims per lane (2 or 4)
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
    const bool live = row < (int64_t)p.num_seqs * p.num_heads;
    int npart = 0;
    bool merge = false;
    if (live) {
        const int s = (int)(row / p.num_heads);
        const dec::Split sp = dec::split_context(__ldg(p.context_lens + s),
                                                 dec::prefix_tokens(p, s), p.max_context_len,
                                                 p.partition_size, p.prefix_partition);
        npart = sp.npre + sp.npart;
        merge = !sp.bad && (sp.pre > 0 || npart > 1);
    }
    pdl_wait_primary();
    if (!merge)
        return;

    const int64_t base = row * p.max_partitions;
    const float* m = p.ws_m + base;
    const float* l = p.ws_l + base;
    uint16_t* out = reinterpret_cast<uint16_t*>(p.out) + row * D + lane * DPL;
    auto store = [&](const float(&acc)[DPL], float inv_l) {
        if constexpr (DPL == 4) {
            const uint32_t w0 = pack2(round_to<QT>(acc[0] * inv_l), round_to<QT>(acc[1] * inv_l));
            const uint32_t w1 = pack2(round_to<QT>(acc[2] * inv_l), round_to<QT>(acc[3] * inv_l));
            *reinterpret_cast<uint2*>(out) = make_uint2(w0, w1);
        } else {
            *reinterpret_cast<uint32_t*>(out) =
                pack2(round_to<QT>(acc[0] * inv_l), round_to<QT>(acc[1] * inv_l));
        }
    };
    if (npart <= kFewParts) {
        // every load first (m, l of partition `lane`; this lane's dims of every
        // partial), so the merge waits for one memory round trip
        float mi = -CUDART_INF_F;
        float li = 0.f;
        if (lane < npart) {
            mi = m[lane];
            li = l[lane];
        }
        float ov[kFewParts][DPL];
        const float* o = p.ws_o + base * D + lane * DPL;
#pragma unroll
        for (int j = 0; j < kFewParts; ++j) {
            if (j < npart) {
                if constexpr (DPL == 4) {
                    const float4 v = *reinterpret_cast<const float4*>(o + (int64_t)j * D);
                    ov[j][0] = v.x, ov[j][1] = v.y, ov[j][2] = v.z, ov[j][3] = v.w;
                } else {
                    const float2 v = *reinterpret_cast<const float2*>(o + (int64_t)j * D);
                    ov[j][0] = v.x, ov[j][1] = v.y;
                }
            }
        }
        float M = mi;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float wl = (M == -CUDART_INF_F || mi == -CUDART_INF_F) ? 0.f : exp2f(mi - M);
        float L = wl * li;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            L += __shfl_xor_sync(0xffffffffu, L, off);
        float acc[DPL];
#pragma unroll
        for (int e = 0; e < DPL; ++e)
            acc[e] = 0.f;
#pragma unroll
        for (int j = 0; j < kFewParts; ++j) {
            const float wj = __shfl_sync(0xffffffffu, wl, j);
            if (j < npart) {
#pragma unroll
                for (int e = 0; e < DPL; ++e)
                    acc[e] = fmaf(wj, ov[j][e], acc[e]);
            }
        }
        store(acc, L > 0.f ? 1.f / L : 0.f);
        return;
    }
    // More partials: lane i keeps m and l of partitions i, i + 32, ... (up to
    // kKeptChunks of them) in registers, so M and the weighted l need one
    // round trip; then each lane accumulates its dims over the partitions
    // kBatch loads at a time (all issued before the first is used).
    constexpr int kKeptChunks = 4;
    constexpr int kBatch = 16;
    float mr[kKeptChunks];
    float lr[kKeptChunks];
    float M = -CUDART_INF_F;
#pragma unroll
    for (int c = 0; c < kKeptChunks; ++c) {
        const int i = lane + 32 * c;
        mr[c] = -CUDART_INF_F;
        lr[c] = 0.f;
        if (i < npart) {
            mr[c] = m[i];
            lr[c] = l[i];
        }
        M = fmaxf(M, mr[c]);
    }
    for (int i = lane + 32 * kKeptChunks; i < npart; i += 32)
        M = fmaxf(M, m[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float wr[kKeptChunks];
    float L = 0.f;
#pragma unroll
    for (int c = 0; c < kKeptChunks; ++c) {
        wr[c] = (M == -CUDART_INF_F || mr[c] == -CUDART_INF_F) ? 0.f : exp2f(mr[c] - M);
        L += wr[c] * lr[c];
    }
    for (int i = lane + 32 * kKeptChunks; i < npart; i += 32) {
        const float mi = m[i];
        if (M != -CUDART_INF_F && mi != -CUDART_INF_F)
            L += exp2f(mi - M) * l[i];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        L += __shfl_xor_sync(0xffffffffu, L, off);

    float acc[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e)
        acc[e] = 0.f;
    const float* o = p.ws_o + base * D + lane * DPL;
    // partitions c0 + [0, n), weight of c0 + j held by lane j
    auto accumulate = [&](int c0, int n, float wl) {
        for (int j0 = 0; j0 < n; j0 += kBatch) {
            float v[kBatch][DPL];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                if (j0 + k < n) {
                    const float* oj = o + (int64_t)(c0 + j0 + k) * D;
                    if constexpr (DPL == 4) {
                        const float4 t = *reinterpret_cast<const float4*>(oj);
                        v[k][0] = t.x, v[k][1] = t.y, v[k][2] = t.z, v[k][3] = t.w;
                    } else {
                        const float2 t = *reinterpret_cast<const float2*>(oj);
                        v[k][0] = t.x, v[k][1] = t.y;
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const float wj = __shfl_sync(0xffffffffu, wl, (j0 + k) & 31);
                if (j0 + k < n) {
#pragma unroll
                    for (int e = 0; e < DPL; ++e)
                        acc[e] = fmaf(wj, v[k][e], acc[e]);
                }
            }
        }
    };
#pragma unroll
    for (int c = 0; c < kKeptChunks; ++c)
        if (32 * c < npart)
            accumulate(32 * c, min(32, npart - 32 * c), wr[c]);
    for (int c0 = 32 * kKeptChunks; c0 < npart; c0 += 32) {
        const int i = c0 + lane;
        float wl = 0.f;
        if (i < npart) {
            const float mi = m[i];
            wl = (M == -CUDART_INF_F || mi == -CUDART_INF_F) ? 0.f : exp2f(mi - M);
        }
        accumulate(c0, min(32, npart - c0), wl);
    }
    store(acc, L > 0.f ? 1.f / L : 0.f);
}

template <int QT>
cudaError_t launch_typed(const ReduceParams& p, cudaLaunchConfig_t& cfg)
{
    if (p.head_dim == 128)
        return cudaLaunchKernelEx(&cfg, lse_reduce_kernel<QT, 128>, p);
    if (p.head_dim == 64)
        return cudaLaunchKernelEx(&cfg, lse_reduce_kernel<QT, 64>, p);
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_lse_reduce(const ReduceParams& p, cudaStream_t stream, bool pdl)
{
    const int64_t rows = (int64_t)p.num_seqs * p.num_heads;
    if (rows <= 0 || p.max_partitions <= 1)
        return cudaSuccess;
    const int64_t ctas = (rows + kRowsPerCta - 1) / kRowsPerCta;
    if (ctas > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kRowsPerCta * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (p.out_dtype == kF16)
        return launch_typed<kF16>(p, cfg);
    if (p.out_dtype == kBF16)
        return launch_typed<kBF16>(p, cfg);
    return cudaErrorNotSupported;
}

}  // namespace pkv
