// decode_common.cuh -- pieces shared by the decode partition kernels: where a
// (sequence, partition) work item stands, and the writes of its result.
#pragma once

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace dec {

constexpr float kNegInf = -__builtin_huge_valf();

__device__ __forceinline__ int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

// Where a (sequence, partition) work item stands.
struct PartitionWork {
    int s;
    int part;
    int t_begin;        // first token of the partition
    int t_end;          // one past its last token
    bool direct;        // context fits one partition: write out, no partials
    bool zero_out;      // write zeros (empty or invalid context) and stop
    bool zero_partial;  // write a neutral partial (table too short) and stop
    bool idle;          // nothing to do
};

// `ctx` is context_lens[s]; `flag` selects the one thread that reports a bad
// context for this item.
__device__ __forceinline__ PartitionWork locate_ctx(const DecodeParams& p, int s, int part, int ctx,
                                                    bool flag)
{
    PartitionWork w{};
    w.s = s;
    w.part = part;
    const bool ctx_oob = ctx < 0 || ctx > p.max_context_len;
    const bool table_short = !ctx_oob && ctx > p.max_blocks_per_seq * p.block_size;
    if ((ctx_oob || table_short) && part == 0 && flag)
        flag_error(p.dev_err, PKV_DEVERR_CONTEXT);
    const int npart = ctx_oob ? 0 : ceil_div_i(ctx, p.partition_size);
    w.direct = npart <= 1;
    if (w.direct) {
        w.idle = part != 0;
        w.zero_out = !w.idle && (ctx_oob || table_short || ctx == 0);
    } else {
        w.idle = part >= npart;
        w.zero_partial = !w.idle && table_short;
    }
    w.t_begin = part * p.partition_size;
    w.t_end = min(ctx, w.t_begin + p.partition_size);
    return w;
}

__device__ __forceinline__ PartitionWork locate(const DecodeParams& p, int s, int part, bool flag)
{
    return locate_ctx(p, s, part, __ldg(p.context_lens + s), flag);
}

__device__ __forceinline__ int64_t partial_row(const DecodeParams& p, int s, int h, int part)
{
    return ((int64_t)s * p.num_heads + h) * p.max_partitions + part;
}

template <int QT>
__device__ __forceinline__ void store_out(const DecodeParams& p, int s, int h, int d, float v)
{
    uint16_t* o = reinterpret_cast<uint16_t*>(p.out);
    o[((int64_t)s * p.num_heads + h) * p.head_dim + d] = round_to<QT>(v);
}

// Writes of an item with no attention to compute, spread over threads
// [0, nthreads) of the caller (tid = this thread's index among them).
template <int QT>
__device__ void write_trivial(const DecodeParams& p, const PartitionWork& w, int head0, int nrows,
                              int tid, int nthreads)
{
    const int D = p.head_dim;
    for (int i = tid; i < nrows * D; i += nthreads) {
        const int h = head0 + i / D;
        const int d = i % D;
        if (w.zero_out) {
            store_out<QT>(p, w.s, h, d, 0.f);
        } else {
            // neutral partial: contributes zero to the merged output
            const int64_t prow = partial_row(p, w.s, h, w.part);
            if (d == 0) {
                p.ws_m[prow] = 0.f;
                p.ws_l[prow] = 1.f;
            }
            p.ws_o[prow * D + d] = 0.f;
        }
    }
}

// Merge of NW per-warp softmax states of `nrows` query heads and the item's
// write.  sm_m / sm_l: [NW][ROWS]; sm_acc: [NW][ROWS][D] (v not yet scaled).
template <int QT, int NW, int ROWS>
__device__ void finish_rows(const DecodeParams& p, const PartitionWork& w, int head0, int nrows,
                            const float* sm_m, const float* sm_l, const float* sm_acc, int tid,
                            int nthreads)
{
    const int D = p.head_dim;
    for (int i = tid; i < nrows * D; i += nthreads) {
        const int row = i / D;
        const int d = i % D;
        float M = kNegInf;
#pragma unroll
        for (int k = 0; k < NW; ++k)
            M = fmaxf(M, sm_m[k * ROWS + row]);
        float L = 0.f;
        float O = 0.f;
        if (M != kNegInf) {
#pragma unroll
            for (int k = 0; k < NW; ++k) {
                const float mk = sm_m[k * ROWS + row];
                if (mk != kNegInf) {
                    const float f = exp2f(mk - M);
                    L += sm_l[k * ROWS + row] * f;
                    O += sm_acc[(k * ROWS + row) * D + d] * f;
                }
            }
        }
        const int h = head0 + row;
        if (w.direct) {
            store_out<QT>(p, w.s, h, d, L > 0.f ? (O / L) * p.v_scale : 0.f);
        } else {
            const int64_t prow = partial_row(p, w.s, h, w.part);
            if (d == 0) {
                p.ws_m[prow] = M;
                p.ws_l[prow] = L;
            }
            p.ws_o[prow * D + d] = O * p.v_scale;
        }
    }
}

}  // namespace dec
}  // namespace pkv
