// decode.cu -- paged decode attention for grouped query heads (one CTA per
// work item), and the choice between it and the streaming kernel.
//
// One CTA handles one partition (partition_size tokens) of one sequence for
// the whole group of query heads that share a KV head.  The grid is ordered
// longest context first, so the hardware dispatches the largest items first.
// Each warp walks a strided subset of the partition's blocks: the physical
// block id comes from the block table
// (「KV 缓存与分页注意力」 §07 块表), the (block, KV head) tile of K and of V is
// read with coalesced 16-byte loads straight into registers, and the warp keeps
// an online softmax (running max and sum, fp32, base 2) with an fp32 P.V
// accumulator.  The warps' states merge through shared memory; the CTA then
// writes either the final output (context within one partition) or its
// partial (m, l, o) for the log-sum-exp reduce kernel (lse_reduce.cu).
#include <cuda_runtime.h>
#include <math_constants.h>

#include "decode_common.cuh"
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

using dec::ceil_div_i;
using dec::kNegInf;
using dec::locate;
using dec::PartitionWork;

// =====================================================================
// Tensor-core kernel for grouped heads (16-bit caches): one CTA per
// (sequence, KV head, partition) computes all G <= 16 query heads of the group
// from one read of each K/V tile, with mma.sync m16n8k16 (fp32 accumulate).
// Fragments below use g = lane / 4 and t = lane % 4.
//
// Scores are computed transposed, S^T = K Q^T, per 16-token sub-block:
// A = K (rows = the 16 tokens, k = head_dim), B = Q^T (n = 8 heads of the
// group per n-tile), so no MMA row is padding when G = 8 or 16.  The head_dim
// index is permuted inside each 32-wide slice so that every fragment register
// comes from one 16-byte load: for k-step 2s+u, thread t's k-columns
// {2t, 2t+1} are dims 32s + 8t + 4u + {0, 1} and {2t+8, 2t+9} are
// 32s + 8t + 4u + {2, 3}; Q and K share the permutation, so every dot product
// is unchanged.  The accumulator gives thread (g, t) the scores of tokens g and
// g + 8 for heads 2t and 2t + 1: the softmax statistics of a head live in the
// eight lanes with the same t.
//
// The output is accumulated transposed too, O^T = V^T P^T: A = V^T (rows =
// head_dim, k = the 16 tokens), B = P^T.  Row m of m-tile j is dim
// 64(j/4) + 8(m%8) + 2(j%4) + m/8, so a thread's A values of one token come
// from one 16-byte load per 64 dims, paired across two tokens with a byte
// permute.  P^T comes from the score accumulators through movmatrix (an 8x8
// transpose of 16-bit elements), and the output accumulator of thread (g, t)
// again belongs to heads 2t and 2t + 1, the heads whose running max it holds.
// bf16 P is split into a high and a low bf16 part (two MMAs) so that the
// weights keep ~16 bits; fp16 P is used as is (11 bits, values in [0, 1]).
// The running max is raised only when some head's block max exceeds it; the
// rescale is skipped otherwise (its factor would be exactly 1).
// =====================================================================
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1,
                                         bool bf16)
{
    if (bf16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

// Transpose of an 8x8 matrix of 16-bit elements held one row pair per lane
// (lane 4i + j holds row i, columns 2j and 2j + 1).
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t reg_of(const uint4& v, int i)
{
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Resident CTAs per SM asked of the compiler: three for one 8-head n-tile
// (168 registers), four in prefix mode (128 registers: the 512 prefix items of
// a parallel-sampling batch then fit one wave), two for 16 heads.
template <int CT, int D, int BS, int NW, int NNT, bool PREFIX>
__global__ void __launch_bounds__(NW * 32, NNT == 1 ? (PREFIX ? 4 : 3) : 2)
    decode_mma_kernel(const DecodeParams p)
{
    constexpr bool kBf16 = (CT == kBF16);
    constexpr int NS = D / 32;          // 32-wide slices of head_dim (QK k-steps / 2)
    constexpr int NH = D / 64;          // 64-wide halves (V loads per token)
    constexpr int NM = D / 16;          // m-tiles of the transposed output
    constexpr int SBB = BS / 16;        // 16-token sub-blocks per block
    constexpr int ROWS = 16;
    static_assert(BS % 16 == 0, "tensor-core path needs 16-token sub-blocks");
    static_assert(D % 64 == 0, "head_dim must be a multiple of 64");
    static_assert(NNT == 1 || NNT == 2, "8 or 16 heads per CTA");

    extern __shared__ __align__(16) float smem[];
    float* sm_m = smem;                        // [NW][16]
    float* sm_l = sm_m + NW * ROWS;            // [NW][16]
    float* sm_acc = sm_l + NW * ROWS;          // [NW][16][D]

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int gq = lane >> 2;
    const int t = lane & 3;
    constexpr int RT = 8 * NNT;                    // rows of one CTA
    const int G = p.group;
    int64_t idx = blockIdx.x;
    const int g = (int)(idx % p.num_kv_heads);
    idx /= p.num_kv_heads;

    // The CTA's rows (query vectors), token range [t_begin, t_end) and block
    // table.  Decode: the G query heads of KV head g of one sequence, over one
    // partition of its context after any shared prefix.  Prefix: rows
    // row0 + [0, RT) of the group's members x G heads, over one partition of
    // the group's shared prefix, read through the first member's table.
    int s = 0;                 // decode: the sequence
    int b0 = 0;                // prefix: the group's first sequence
    int row0 = 0;
    int nrows = G;
    int t_begin = 0;
    int t_end = 0;
    int slot = 0;
    bool direct = false;
    const int32_t* table = nullptr;
    if constexpr (PREFIX) {
        const int ntiles = ceil_div_i(p.max_group_size * G, RT);
        const int tile = (int)(idx % ntiles);
        idx /= ntiles;
        const int grp = (int)(idx % p.num_groups);
        const int chunk = (int)(idx / p.num_groups);
        b0 = __ldg(p.grp_begin + grp);
        const int b1 = __ldg(p.grp_begin + grp + 1);
        const int blocks = __ldg(p.grp_prefix_blocks + grp);
        const bool first = g == 0 && tile == 0 && chunk == 0 && threadIdx.x == 0;
        if (b0 < 0 || b1 < b0 || b1 > p.num_seqs || blocks < 0 ||
            blocks > min(p.max_prefix_blocks, p.max_blocks_per_seq)) {
            if (first)
                flag_error(p.dev_err, PKV_DEVERR_PREFIX);
            return;
        }
        const int nmem = min(b1 - b0, p.max_group_size);
        // every member's table must hold the first member's prefix blocks
        if (g == 0 && tile == 0 && chunk == 0) {
            const int32_t* lead = p.block_tables + (int64_t)b0 * p.max_blocks_per_seq;
            for (int i = threadIdx.x; i < (nmem - 1) * blocks; i += blockDim.x) {
                const int m = 1 + i / blocks;
                const int b = i % blocks;
                if (__ldg(lead + (int64_t)m * p.max_blocks_per_seq + b) != __ldg(lead + b))
                    flag_error(p.dev_err, PKV_DEVERR_PREFIX);
            }
        }
        t_begin = chunk * p.prefix_partition;
        t_end = min(blocks * BS, t_begin + p.prefix_partition);
        row0 = tile * RT;
        nrows = min(RT, nmem * G - row0);
        if (t_begin >= t_end || nrows <= 0)
            return;
        slot = chunk;
        table = p.block_tables + (int64_t)b0 * p.max_blocks_per_seq + t_begin / BS;
        pdl_launch_dependents();
    } else {
        const int srank = (int)(idx % p.num_seqs);
        const int part = (int)(idx / p.num_seqs);
        // grid position -> sequence: longest context first (ties by index)
        // for batches of up to 128 sequences, in order otherwise
        s = srank;
        if (p.num_seqs <= 128) {
            __shared__ int sh_ctx[128];
            __shared__ int sh_seq;
            for (int i = threadIdx.x; i < p.num_seqs; i += blockDim.x)
                sh_ctx[i] = __ldg(p.context_lens + i);
            __syncthreads();
            for (int i = threadIdx.x; i < p.num_seqs; i += blockDim.x) {
                const int ci = sh_ctx[i];
                int rank = 0;
                for (int j = 0; j < p.num_seqs; ++j)
                    rank += (sh_ctx[j] > ci) || (sh_ctx[j] == ci && j < i);
                if (rank == srank)
                    sh_seq = i;
            }
            __syncthreads();
            s = sh_seq;
        }

        pdl_launch_dependents();

        const PartitionWork w = locate(p, s, part, threadIdx.x == 0);
        if (w.idle || w.zero_out || w.zero_partial) {
            if (!w.idle)
                dec::write_trivial<CT>(p, w, g * G, G, threadIdx.x, blockDim.x);
            if (p.wait_prior && threadIdx.x == 0)
                pdl_wait_primary();
            return;
        }
        t_begin = w.t_begin;
        t_end = w.t_end;
        table = p.block_tables + (int64_t)s * p.max_blocks_per_seq + t_begin / BS;
    }
    // row r -> (sequence, query head)
    auto row_of = [&](int r) -> int2 {
        if constexpr (PREFIX) {
            const int rho = row0 + r;
            return make_int2(b0 + rho / G, g * G + rho % G);
        } else {
            return make_int2(s, g * G + r);
        }
    };

    // Q^T fragments: rows gq (+ 8 for the second n-tile), zero past nrows
    // kept in shared memory as sq[n][i][lane] (each lane reads back its own
    // 16 bytes: conflict-free) rather than in registers, which the K/V loads
    // of the block loop need
    uint4* sq = reinterpret_cast<uint4*>(sm_acc + NW * ROWS * D);     // [NNT][NS][32]
    for (int i = threadIdx.x; i < NNT * NS * 32; i += blockDim.x) {
        const int ln = i & 31;
        const int r = (ln >> 2) + 8 * (i / (NS * 32));
        const int sl = (i >> 5) % NS;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < nrows) {
            const int2 sh = row_of(r);
            v = ld_ro(reinterpret_cast<const char*>(p.q) +
                      (((int64_t)sh.x * p.num_heads + sh.y) * D + 32 * sl + 8 * (ln & 3)) * 2);
        }
        sq[i] = v;
    }
    __syncthreads();

    const int nblk = ceil_div_i(t_end - t_begin, BS);
    const int64_t tile_elems = (int64_t)BS * D;
    const int64_t block_stride = (int64_t)p.num_kv_heads * tile_elems;
    const char* kbase = reinterpret_cast<const char*>(p.k_cache) + (int64_t)g * tile_elems * 2;
    const char* vbase = reinterpret_cast<const char*>(p.v_cache) + (int64_t)g * tile_elems * 2;
    const float qk = p.qk_scale_log2;

    // output accumulators (m-tile j, head tile n) and per-head softmax state
    // of heads 8n + 2t + {0, 1}
    float acc[NM][NNT][4];
#pragma unroll
    for (int j = 0; j < NM; ++j)
#pragma unroll
        for (int n = 0; n < NNT; ++n)
            acc[j][n][0] = acc[j][n][1] = acc[j][n][2] = acc[j][n][3] = 0.f;
    float m_h[NNT][2];
    float l_h[NNT][2];
#pragma unroll
    for (int n = 0; n < NNT; ++n)
        m_h[n][0] = m_h[n][1] = kNegInf, l_h[n][0] = l_h[n][1] = 0.f;

    // The warp walks blocks warp, warp + NW, ... of the partition, one
    // 16-token sub-block at a time.  The loop body is unrolled twice, which
    // lets the compiler issue the next sub-block's loads early.
    const int my_blocks = nblk > warp ? ceil_div_i(nblk - warp, NW) : 0;
    const int nsub = my_blocks * SBB;
    int cur_chunk = -1;
    int my_entry = -1;
    auto phys_of = [&](int it) -> int {          // warp-uniform
        const int ch = it >> 5;
        if (ch != cur_chunk) {
            cur_chunk = ch;
            const int bi = warp + (ch * 32 + lane) * NW;
            my_entry = bi < nblk ? __ldg(table + bi) : -1;
        }
        return __shfl_sync(0xffffffffu, my_entry, it & 31);
    };
    // byte offset of sub-block q inside the caches, or -1 for a bad block id
    auto sub_tile = [&](int q) -> int64_t {
        const int phys = phys_of(q / SBB);
        if (phys < 0 || (int64_t)phys >= p.num_blocks) {
            if (lane == 0 && q % SBB == 0)
                flag_error(p.dev_err, PKV_DEVERR_BLOCK_ID);
            return -1;
        }
        return ((int64_t)phys * block_stride + (int64_t)(q % SBB) * 16 * D) * 2;
    };
    auto load_k = [&](int64_t off, uint4(&k)[2][NS]) {
        const char* kt = kbase + off;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
            for (int i = 0; i < NS; ++i)
                k[hf][i] = ld_stream(kt + ((hf * 8 + gq) * D + 32 * i + 8 * t) * 2);
    };

    auto step = [&](int q, int64_t& off, uint4(&kc)[2][NS]) {
        const int i = warp + (q / SBB) * NW;                  // block of the partition
        const int tb = t_begin + i * BS + (q % SBB) * 16;   // first token of the sub-block
        const bool live = off >= 0 && tb < t_end;           // warp-uniform
        // V rows of tokens 2t, 2t + 1, 2t + 8, 2t + 9: dims 64 hv + 8 gq + [0, 8)
        uint4 vc[4][NH];
        float sc[NNT][4];
        if (live) {
            load_k(off, kc);
            const char* vt = vbase + off;
#pragma unroll
            for (int tk = 0; tk < 4; ++tk)
#pragma unroll
                for (int hv = 0; hv < NH; ++hv)
                    vc[tk][hv] = ld_stream(
                        vt + ((2 * t + (tk & 1) + 8 * (tk >> 1)) * D + 64 * hv + 8 * gq) * 2);
            // S^T = K Q^T: rows = tokens tb + gq, tb + gq + 8
#pragma unroll
            for (int n = 0; n < NNT; ++n)
                sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
            for (int i2 = 0; i2 < NS; ++i2) {
                uint4 qv[NNT];
#pragma unroll
                for (int n = 0; n < NNT; ++n)
                    qv[n] = ld_shared16(sq + (n * NS + i2) * 32 + lane);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const uint32_t a[4] = {reg_of(kc[0][i2], 2 * u), reg_of(kc[1][i2], 2 * u),
                                           reg_of(kc[0][i2], 2 * u + 1),
                                           reg_of(kc[1][i2], 2 * u + 1)};
#pragma unroll
                    for (int n = 0; n < NNT; ++n)
                        mma16816(sc[n], a, reg_of(qv[n], 2 * u), reg_of(qv[n], 2 * u + 1),
                                 kBf16);
                }
            }
        }
        const int64_t off_n = q + 1 < nsub ? sub_tile(q + 1) : -1;
        if (live) {
            // online softmax (base 2); sc[n][e] is token tb + gq + 8 (e >> 1),
            // head 8n + 2t + (e & 1)
            float x[NNT][4];
            float mn[NNT][2];
            bool raise = false;
#pragma unroll
            for (int n = 0; n < NNT; ++n) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    x[n][e] = (tb + gq + 8 * (e >> 1) < t_end) ? sc[n][e] * qk : kNegInf;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float mx = fmaxf(x[n][h], x[n][h + 2]);
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    mn[n][h] = fmaxf(m_h[n][h], mx);
                    raise |= mn[n][h] > m_h[n][h];
                }
            }
            if (__any_sync(0xffffffffu, raise)) {
                float al[NNT][2];
#pragma unroll
                for (int n = 0; n < NNT; ++n)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        al[n][h] = exp2f(m_h[n][h] - mn[n][h]);
                        m_h[n][h] = mn[n][h];
                        l_h[n][h] *= al[n][h];
                    }
#pragma unroll
                for (int j = 0; j < NM; ++j)
#pragma unroll
                    for (int n = 0; n < NNT; ++n)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            acc[j][n][e] *= al[n][e & 1];
            }
            float pr[NNT][4];
#pragma unroll
            for (int n = 0; n < NNT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    pr[n][e] = x[n][e] == kNegInf ? 0.f : exp2f(x[n][e] - m_h[n][e & 1]);
                    l_h[n][e & 1] += pr[n][e];
                }

            // tokens past the context contribute p = 0; clear their V so that
            // whatever bits sit in those slots cannot make NaN
#pragma unroll
            for (int tk = 0; tk < 4; ++tk)
                if (tb + 2 * t + (tk & 1) + 8 * (tk >> 1) >= t_end)
#pragma unroll
                    for (int hv = 0; hv < NH; ++hv)
                        vc[tk][hv] = make_uint4(0, 0, 0, 0);

            // P^T fragments: rows gq, gq + 8 of the accumulator are tokens, so
            // the 8x8 transposes give lane (gq, t) head gq, tokens 2t, 2t + 1
            // (+ 8 for the second register)
            uint32_t bh[NNT][2];
            uint32_t bl[NNT][2];
#pragma unroll
            for (int n = 0; n < NNT; ++n)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const float v0 = pr[n][2 * hf];
                    const float v1 = pr[n][2 * hf + 1];
                    if constexpr (kBf16) {
                        const uint16_t h0 = round_to<kBF16>(v0), h1 = round_to<kBF16>(v1);
                        const float r0 = v0 - __uint_as_float((uint32_t)h0 << 16);
                        const float r1 = v1 - __uint_as_float((uint32_t)h1 << 16);
                        bh[n][hf] = transpose8x8(pack2(h0, h1));
                        bl[n][hf] =
                            transpose8x8(pack2(round_to<kBF16>(r0), round_to<kBF16>(r1)));
                    } else {
                        bh[n][hf] = transpose8x8(pack2(round_to<kF16>(v0), round_to<kF16>(v1)));
                        bl[n][hf] = 0u;
                    }
                }

            // O^T += V^T P^T
#pragma unroll
            for (int j = 0; j < NM; ++j) {
                const int hv = j >> 2;
                const int e = j & 3;
                const uint32_t lo0 = reg_of(vc[0][hv], e), lo1 = reg_of(vc[1][hv], e);
                const uint32_t hi0 = reg_of(vc[2][hv], e), hi1 = reg_of(vc[3][hv], e);
                const uint32_t a[4] = {__byte_perm(lo0, lo1, 0x5410), __byte_perm(lo0, lo1, 0x7632),
                                       __byte_perm(hi0, hi1, 0x5410), __byte_perm(hi0, hi1, 0x7632)};
#pragma unroll
                for (int n = 0; n < NNT; ++n) {
                    mma16816(acc[j][n], a, bh[n][0], bh[n][1], kBf16);
                    if constexpr (kBf16)
                        mma16816(acc[j][n], a, bl[n][0], bl[n][1], kBf16);
                }
            }
        }
        off = off_n;
    };

    uint4 kf[2][NS];
    int64_t off = nsub > 0 ? sub_tile(0) : -1;
    for (int q = 0; q < nsub; q += 2) {
        step(q, off, kf);
        if (q + 1 < nsub)
            step(q + 1, off, kf);
    }

    // head sums over the eight lanes of a head
#pragma unroll
    for (int n = 0; n < NNT; ++n)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float l = l_h[n][h];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            l_h[n][h] = l;
        }
    if (gq == 0) {
#pragma unroll
        for (int n = 0; n < NNT; ++n)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                sm_m[warp * ROWS + 8 * n + 2 * t + h] = m_h[n][h];
                sm_l[warp * ROWS + 8 * n + 2 * t + h] = l_h[n][h];
            }
    }
    // accumulator (j, n, e): head 8n + 2t + (e & 1),
    // dim 64 (j / 4) + 8 gq + 2 (j % 4) + (e >> 1)
#pragma unroll
    for (int j = 0; j < NM; ++j)
#pragma unroll
        for (int n = 0; n < NNT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = 8 * n + 2 * t + (e & 1);
                const int d = 64 * (j >> 2) + 8 * gq + 2 * (j & 3) + (e >> 1);
                sm_acc[(warp * ROWS + row) * D + d] = acc[j][n][e];
            }
    if constexpr (!PREFIX) {
        // where this item's result goes (recomputed: nothing stays live
        // across the loop for it)
        const PartitionWork w = locate(p, s, (int)(blockIdx.x / p.num_kv_heads / p.num_seqs),
                                       false);
        slot = w.slot;
        direct = w.direct;
    }
    __syncthreads();
    dec::finish_rows_map<CT, NW, ROWS>(p, direct, slot, nrows, row_of, sm_m, sm_l, sm_acc,
                                       threadIdx.x, blockDim.x);
    if (!PREFIX && p.wait_prior && threadIdx.x == 0)
        pdl_wait_primary();
}

// ------------------------------------------------------------------ dispatch

constexpr int kWarps = 4;

template <int CT, int D, int BS, int NNT, bool PREFIX>
cudaError_t run_mma_heads(const DecodeParams& p, dim3 grid, cudaStream_t stream)
{
    // merge area (per warp 16 row maxima, 16 row sums and a 16 x D
    // accumulator), then the Q fragments (NNT x D/32 x 32 lanes x 16 bytes)
    constexpr size_t smem = sizeof(float) * (2 * kWarps * 16 + kWarps * 16 * D) + NNT * D * 16;
    auto kern = decode_mma_kernel<CT, D, BS, kWarps, NNT, PREFIX>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (!PREFIX && p.wait_prior) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

// rows per CTA: 8 when they fit, else 16
template <int CT, int D, int BS, bool PREFIX>
cudaError_t run_mma(const DecodeParams& p, int rows, dim3 grid, cudaStream_t stream)
{
    return rows > 8 ? run_mma_heads<CT, D, BS, 2, PREFIX>(p, grid, stream)
                    : run_mma_heads<CT, D, BS, 1, PREFIX>(p, grid, stream);
}

template <int CT, bool PREFIX>
cudaError_t mma_shape(const DecodeParams& p, int rows, dim3 grid, cudaStream_t st)
{
    if (p.head_dim == 64 && p.block_size == 16) return run_mma<CT, 64, 16, PREFIX>(p, rows, grid, st);
    if (p.head_dim == 64 && p.block_size == 32) return run_mma<CT, 64, 32, PREFIX>(p, rows, grid, st);
    if (p.head_dim == 128 && p.block_size == 16) return run_mma<CT, 128, 16, PREFIX>(p, rows, grid, st);
    if (p.head_dim == 128 && p.block_size == 32) return run_mma<CT, 128, 32, PREFIX>(p, rows, grid, st);
    return cudaErrorNotSupported;
}

bool use_mma(const DecodeParams& p)
{
    return p.group >= 2 && p.group <= 16 && p.cache_dtype != kE4M3 &&
           p.cache_dtype == p.q_dtype && (p.block_size % 16) == 0;
}

}  // namespace

bool decode_shape_supported(int cache_dtype, int q_dtype, int head_dim, int block_size)
{
    if (head_dim != 64 && head_dim != 128)
        return false;
    if (block_size != 8 && block_size != 16 && block_size != 32)
        return false;
    if (q_dtype != kF16 && q_dtype != kBF16)
        return false;
    if (cache_dtype == kE4M3)
        return true;
    return cache_dtype == q_dtype;
}

cudaError_t launch_decode_partitions(const DecodeParams& p, cudaStream_t stream)
{
    if (!decode_shape_supported(p.cache_dtype, p.q_dtype, p.head_dim, p.block_size))
        return cudaErrorNotSupported;
    const bool mma = use_mma(p);
    const int64_t heads = mma ? p.num_kv_heads : p.num_heads;
    const int64_t ctas = (int64_t)p.grid_partitions * p.num_seqs * heads;
    if (ctas <= 0)
        return cudaSuccess;
    if (ctas > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)ctas);
    // single-head items: the persistent streaming kernel (decode_stream.cu);
    // grouped heads: the one-CTA-per-item tensor-core kernel above
    if (!mma)
        return launch_decode_stream(p, false, stream);
    return p.cache_dtype == kF16 ? mma_shape<kF16, false>(p, p.group, grid, stream)
                                 : mma_shape<kBF16, false>(p, p.group, grid, stream);
}

bool prefix_kernel_supported(int cache_dtype, int q_dtype, int head_dim, int block_size,
                             int group)
{
    return (head_dim == 64 || head_dim == 128) && (block_size == 16 || block_size == 32) &&
           (cache_dtype == kF16 || cache_dtype == kBF16) && cache_dtype == q_dtype &&
           group >= 1 && group <= 16;
}

cudaError_t launch_decode_prefix(const DecodeParams& p, cudaStream_t stream)
{
    if (!prefix_kernel_supported(p.cache_dtype, p.q_dtype, p.head_dim, p.block_size, p.group))
        return cudaErrorNotSupported;
    if (p.grp_begin == nullptr || p.num_groups <= 0 || p.max_group_size <= 0 ||
        p.max_prefix_blocks <= 0)
        return cudaSuccess;
    // members x heads of a KV head, in tiles of 8 or 16 rows
    const int64_t rows = (int64_t)p.max_group_size * p.group;
    const int rt = rows > 8 ? 16 : 8;
    const int64_t tiles = (rows + rt - 1) / rt;
    if (p.prefix_partition <= 0)
        return cudaErrorInvalidValue;
    const int64_t chunks = ((int64_t)p.max_prefix_blocks * p.block_size + p.prefix_partition - 1) /
                           p.prefix_partition;
    const int64_t ctas = chunks * p.num_groups * tiles * p.num_kv_heads;
    if (ctas > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)ctas);
    const int r = (int)(rows > 8 ? 16 : 8);
    return p.cache_dtype == kF16 ? mma_shape<kF16, true>(p, r, grid, stream)
                                 : mma_shape<kBF16, true>(p, r, grid, stream);
}

}  // namespace pkv
