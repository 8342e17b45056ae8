// decode_common.cuh -- pieces shared by the decode partition kernels: where a
// (sequence, partition) work item stands, and the writes of its result.
#pragma once

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace dec {

constexpr float kNegInf = -__builtin_huge_valf();

__device__ __forceinline__ int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

// Shared-prefix tokens of sequence s: grp_prefix_blocks[i] * block_size for
// the group i holding s, 0 without groups, -1 when the group's entry cannot be
// used (a negative or too long prefix, or s beyond the member count the
// prefix kernel covers).  PT is DecodeParams or ReduceParams.
template <class PT>
__device__ __forceinline__ int prefix_tokens(const PT& p, int s)
{
    if (p.grp_begin == nullptr || p.num_groups <= 0)
        return 0;
    int lo = 0;
    int hi = p.num_groups;                 // the last i with grp_begin[i] <= s
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(p.grp_begin + mid) <= s)
            lo = mid;
        else
            hi = mid;
    }
    const int blocks = __ldg(p.grp_prefix_blocks + lo);
    if (blocks == 0)
        return 0;
    const int b0 = __ldg(p.grp_begin + lo);
    if (blocks < 0 || blocks > p.max_prefix_blocks || s < b0 || s - b0 >= p.max_group_size)
        return -1;
    return blocks * p.block_size;
}

// How the context of one sequence splits into partials: `npre` partitions of
// prefix_partition tokens of the shared prefix (written by the prefix kernel)
// come first, then `npart` partitions of partition_size tokens of the rest of
// the context.  `bad` marks a context length or prefix that cannot be used:
// the sequence's output is zero.
struct Split {
    int pre;            // prefix tokens
    int npre;
    int npart;
    bool bad;
};

__device__ __forceinline__ Split split_context(int ctx, int pre, int max_context_len,
                                               int partition_size, int prefix_partition)
{
    Split sp{};
    sp.bad = ctx < 0 || ctx > max_context_len || pre < 0 || pre > ctx;
    if (!sp.bad) {
        sp.pre = pre;
        sp.npre = pre > 0 ? ceil_div_i(pre, prefix_partition) : 0;
        sp.npart = ceil_div_i(ctx - pre, partition_size);
    }
    return sp;
}

// Where a (sequence, partition) work item stands.
struct PartitionWork {
    int s;
    int slot;           // its partial's index among the sequence's partials
    int t_begin;        // first token of the partition
    int t_end;          // one past its last token
    bool direct;        // context fits one partition: write out, no partials
    bool zero_out;      // write zeros (empty or invalid context) and stop
    bool zero_partial;  // write a neutral partial (table too short) and stop
    bool idle;          // nothing to do
};

// Partition `part` of the part of sequence s's context after its shared
// prefix.  `ctx` is context_lens[s]; `flag` selects the one thread that
// reports a bad context for this item.
__device__ __forceinline__ PartitionWork locate_ctx(const DecodeParams& p, int s, int part, int ctx,
                                                    bool flag)
{
    PartitionWork w{};
    w.s = s;
    const Split sp = split_context(ctx, prefix_tokens(p, s), p.max_context_len,
                                   p.partition_size, p.prefix_partition);
    const bool table_short = !sp.bad && ctx > p.max_blocks_per_seq * p.block_size;
    if ((sp.bad || table_short) && part == 0 && flag)
        flag_error(p.dev_err, PKV_DEVERR_CONTEXT);
    w.direct = sp.pre == 0 && sp.npart <= 1;
    if (w.direct) {
        w.idle = part != 0;
        w.zero_out = !w.idle && (sp.bad || table_short || ctx == 0);
    } else {
        w.idle = part >= sp.npart;
        w.zero_partial = !w.idle && table_short;
    }
    w.slot = sp.npre + part;
    w.t_begin = sp.pre + part * p.partition_size;
    w.t_end = min(ctx, w.t_begin + p.partition_size);
    return w;
}

__device__ __forceinline__ PartitionWork locate(const DecodeParams& p, int s, int part, bool flag)
{
    return locate_ctx(p, s, part, __ldg(p.context_lens + s), flag);
}

__device__ __forceinline__ int64_t partial_row(const DecodeParams& p, int s, int h, int slot)
{
    return ((int64_t)s * p.num_heads + h) * p.max_partitions + slot;
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
            const int64_t prow = partial_row(p, w.s, h, w.slot);
            if (d == 0) {
                p.ws_m[prow] = 0.f;
                p.ws_l[prow] = 1.f;
            }
            p.ws_o[prow * D + d] = 0.f;
        }
    }
}

// Merge of NW per-warp softmax states of `nrows` rows and their write.
// sm_m / sm_l: [NW][ROWS]; sm_acc: [NW][ROWS][D] (v not yet scaled).  Row r
// is query head rowmap(r).y of sequence rowmap(r).x; `direct` writes the
// output, otherwise the partial at index `slot`.
template <int QT, int NW, int ROWS, class RowMap>
__device__ void finish_rows_map(const DecodeParams& p, bool direct, int slot, int nrows,
                                RowMap rowmap, const float* sm_m, const float* sm_l,
                                const float* sm_acc, int tid, int nthreads)
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
        const int2 sh = rowmap(row);
        if (direct) {
            store_out<QT>(p, sh.x, sh.y, d, L > 0.f ? (O / L) * p.v_scale : 0.f);
        } else {
            const int64_t prow = partial_row(p, sh.x, sh.y, slot);
            if (d == 0) {
                p.ws_m[prow] = M;
                p.ws_l[prow] = L;
            }
            p.ws_o[prow * D + d] = O * p.v_scale;
        }
    }
}

// The same for the query heads head0 + [0, nrows) of one work item.
template <int QT, int NW, int ROWS>
__device__ void finish_rows(const DecodeParams& p, const PartitionWork& w, int head0, int nrows,
                            const float* sm_m, const float* sm_l, const float* sm_acc, int tid,
                            int nthreads)
{
    const int s = w.s;
    finish_rows_map<QT, NW, ROWS>(
        p, w.direct, w.slot, nrows, [=](int r) { return make_int2(s, head0 + r); }, sm_m, sm_l,
        sm_acc, tid, nthreads);
}

}  // namespace dec
}  // namespace pkv
