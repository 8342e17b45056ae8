// decode.cu -- paged decode attention, split-context partition kernels.
//
// One CTA handles one partition (partition_size tokens) of one sequence, for
// one query head (CUDA-core kernel) or for the whole group of query heads that
// share a KV head (tensor-core kernel).  Each warp walks a strided subset of
// the partition's blocks: the physical block id comes from the block table
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
// CUDA-core kernel: one query head per CTA.
//
// Lane layout inside a warp for one (block, KV head) tile of BS x D elements:
// the tile is BS*D*C bytes = NV 16-byte vectors per lane; vector j of lane l is
// at byte (j*32 + l)*16, i.e. token j*TPI + l/RV, elements (l%RV)*EPV ... +EPV.
// Every load instruction covers 512 contiguous bytes.
// =====================================================================
template <int CT, int QT, int D, int BS, int NW>
__global__ void __launch_bounds__(NW * 32, 4) decode_simt_kernel(const DecodeParams p)
{
    constexpr int C = Elem<CT>::bytes;
    constexpr int EPV = 16 / C;          // elements per 16-byte vector
    constexpr int RV = D / EPV;          // vectors per token row
    constexpr int TPI = 32 / RV;         // tokens per warp-wide load
    constexpr int NV = BS / TPI;         // vectors per lane per tile
    static_assert(RV >= 1 && RV <= 32 && 32 % RV == 0, "row must split evenly over lanes");
    static_assert(BS % TPI == 0, "block must cover whole warp loads");
    constexpr int ROWS = 1;

    __shared__ float sm_m[NW * ROWS];
    __shared__ float sm_l[NW * ROWS];
    __shared__ __align__(16) float sm_acc[NW * ROWS * D];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    int64_t idx = blockIdx.x;
    const int h = (int)(idx % p.num_heads);
    idx /= p.num_heads;
    const int s = (int)(idx % p.num_seqs);
    const int part = (int)(idx / p.num_seqs);

    pdl_launch_dependents();

    const PartitionWork w = locate(p, s, part, threadIdx.x == 0);
    if (w.idle)
        return;
    if (w.zero_out || w.zero_partial) {
        dec::write_trivial<QT>(p, w, h, 1, threadIdx.x, blockDim.x);
        return;
    }

    const int g = h / p.group;
    const int dchunk = lane % RV;
    const int tsub = lane / RV;

    // query slice of this lane, pre-multiplied by scale * log2(e) * k_scale
    float qf[EPV];
    {
        const char* qrow = reinterpret_cast<const char*>(p.q) +
                           (((int64_t)s * p.num_heads + h) * D + dchunk * EPV) * 2;
#pragma unroll
        for (int i = 0; i < EPV / 8; ++i) {
            const uint4 v = ld_ro(qrow + 16 * i);
            unpack_vec<QT>(v, qf + 8 * i);
        }
#pragma unroll
        for (int e = 0; e < EPV; ++e)
            qf[e] *= p.qk_scale_log2;
    }

    const int nblk = ceil_div_i(w.t_end - w.t_begin, BS);
    const int blk0 = w.t_begin / BS;
    const int32_t* table = p.block_tables + (int64_t)s * p.max_blocks_per_seq + blk0;
    const int64_t tile_elems = (int64_t)BS * D;
    const int64_t head_off = (int64_t)g * tile_elems;
    const int64_t block_stride = (int64_t)p.num_kv_heads * tile_elems;
    const char* kbase = reinterpret_cast<const char*>(p.k_cache) + head_off * C;
    const char* vbase = reinterpret_cast<const char*>(p.v_cache) + head_off * C;

    float m_run = kNegInf;
    float l_run = 0.f;
    float acc[EPV];
#pragma unroll
    for (int e = 0; e < EPV; ++e)
        acc[e] = 0.f;

    // this warp's blocks: i = warp, warp + NW, ...; table entries prefetched
    // 32 at a time into one register per lane
    for (int chunk = 0; warp + chunk * 32 * NW < nblk; ++chunk) {
        const int first = warp + chunk * 32 * NW;
        int my_entry = -1;
        {
            const int i = first + lane * NW;
            if (i < nblk)
                my_entry = __ldg(table + i);
        }
        const int iters = min(32, ceil_div_i(nblk - first, NW));
        for (int it = 0; it < iters; ++it) {
            const int i = first + it * NW;
            const int phys = __shfl_sync(0xffffffffu, my_entry, it);
            if (phys < 0 || (int64_t)phys >= p.num_blocks) {
                if (lane == 0)
                    flag_error(p.dev_err, PKV_DEVERR_BLOCK_ID);
                continue;
            }
            const char* kt = kbase + (int64_t)phys * block_stride * C;
            const char* vt = vbase + (int64_t)phys * block_stride * C;
            uint4 kv[NV];
            uint4 vv[NV];
#pragma unroll
            for (int j = 0; j < NV; ++j)
                kv[j] = ld_stream(kt + (j * 32 + lane) * 16);
#pragma unroll
            for (int j = 0; j < NV; ++j)
                vv[j] = ld_stream(vt + (j * 32 + lane) * 16);

            const int tok0 = w.t_begin + i * BS + tsub;     // token of vector 0
            float x[NV];
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                float kf[EPV];
                unpack_vec<CT>(kv[j], kf);
                float dot = 0.f;
#pragma unroll
                for (int e = 0; e < EPV; ++e)
                    dot = fmaf(qf[e], kf[e], dot);
#pragma unroll
                for (int off = RV / 2; off > 0; off >>= 1)
                    dot += __shfl_xor_sync(0xffffffffu, dot, off);
                x[j] = (tok0 + j * TPI < w.t_end) ? dot : kNegInf;
            }
            float mx = x[0];
#pragma unroll
            for (int j = 1; j < NV; ++j)
                mx = fmaxf(mx, x[j]);
#pragma unroll
            for (int off = RV; off < 32; off <<= 1)
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_new = fmaxf(m_run, mx);
            const float alpha = exp2f(m_run - m_new);
            m_run = m_new;
            l_run *= alpha;
#pragma unroll
            for (int e = 0; e < EPV; ++e)
                acc[e] *= alpha;
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                if (tok0 + j * TPI < w.t_end) {
                    const float pj = exp2f(x[j] - m_new);
                    l_run += pj;
                    float vf[EPV];
                    unpack_vec<CT>(vv[j], vf);
#pragma unroll
                    for (int e = 0; e < EPV; ++e)
                        acc[e] = fmaf(pj, vf[e], acc[e]);
                }
            }
        }
    }

    // sum over the lanes that share this lane's d-chunk (different tokens)
#pragma unroll
    for (int off = RV; off < 32; off <<= 1) {
        l_run += __shfl_xor_sync(0xffffffffu, l_run, off);
#pragma unroll
        for (int e = 0; e < EPV; ++e)
            acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
    }
    if (lane < RV) {
#pragma unroll
        for (int e = 0; e < EPV; ++e)
            sm_acc[warp * D + lane * EPV + e] = acc[e];
    }
    if (lane == 0) {
        sm_m[warp] = m_run;
        sm_l[warp] = l_run;
    }
    __syncthreads();
    dec::finish_rows<QT, NW, ROWS>(p, w, h, 1, sm_m, sm_l, sm_acc, threadIdx.x, blockDim.x);
}

// =====================================================================
// Tensor-core kernel for grouped heads (16-bit caches): one CTA per
// (sequence, KV head, partition) computes all G <= 16 query heads of the group
// from one read of each K/V tile, with mma.sync m16n8k16 (fp32 accumulate).
//
// S = Q K^T per 16-token sub-block: A = Q (rows = heads, padded to 16),
// B = K^T (8 tokens per n-tile), K-dim = head_dim.  The head_dim index is
// permuted inside each 32-wide slice so that every fragment register comes
// from one 16-byte load: thread (r = lane/4, c = lane%4) holds, for k-step
// 2s'+u, dims 32s' + 8c + 4u + {0,1} and + {2,3}; the same permutation applies
// to Q and K, which leaves every dot product unchanged.
// O = P V: A = P straight from the S accumulators (rows = heads, k = tokens),
// B = V with output column n of n-tile j at dim 64(j/8) + 8n + j%8, so that a
// thread's B values of one token come from one 16-byte load per 64 dims; the
// accumulator of thread (r, c) then holds dims 64(j/8) + 16c + {0..15}.
// bf16 P is split into a high and a low bf16 part (two MMAs) so that the
// weights keep ~16 bits; fp16 P is used as is (11 bits, values in [0, 1]).
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

template <int DT>
__device__ __forceinline__ uint32_t pack_f32x2(float lo, float hi)
{
    return pack2(round_to<DT>(lo), round_to<DT>(hi));
}

__device__ __forceinline__ uint32_t reg_of(const uint4& v, int i)
{
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

template <int CT, int D, int BS, int NW, bool TWO_ROWS>
__global__ void __launch_bounds__(NW * 32, 2) decode_mma_kernel(const DecodeParams p)
{
    constexpr bool kBf16 = (CT == kBF16);
    constexpr int NS = D / 32;          // 32-wide slices of head_dim (QK k-steps / 2)
    constexpr int NH = D / 64;          // 64-wide halves (V loads per token)
    constexpr int NT = D / 8;           // n-tiles of the output
    constexpr int ROWS = 16;
    static_assert(BS % 16 == 0, "tensor-core path needs 16-token sub-blocks");
    static_assert(D % 64 == 0, "head_dim must be a multiple of 64");

    extern __shared__ __align__(16) float smem[];
    float* sm_m = smem;                        // [NW][16]
    float* sm_l = sm_m + NW * ROWS;            // [NW][16]
    float* sm_acc = sm_l + NW * ROWS;          // [NW][16][D]

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int r = lane >> 2;
    const int c = lane & 3;
    int64_t idx = blockIdx.x;
    const int g = (int)(idx % p.num_kv_heads);
    idx /= p.num_kv_heads;
    const int s = (int)(idx % p.num_seqs);
    const int part = (int)(idx / p.num_seqs);
    const int G = p.group;
    const int head0 = g * G;

    pdl_launch_dependents();

    const PartitionWork w = locate(p, s, part, threadIdx.x == 0);
    if (w.idle)
        return;
    if (w.zero_out || w.zero_partial) {
        dec::write_trivial<CT>(p, w, head0, G, threadIdx.x, blockDim.x);
        return;
    }

    // Q fragments: rows r and r + 8 of the group (zero past G)
    uint4 qa[NS];
    uint4 qb[TWO_ROWS ? NS : 1];
    {
        const char* qbase = reinterpret_cast<const char*>(p.q) +
                            ((int64_t)s * p.num_heads + head0) * D * 2;
#pragma unroll
        for (int i = 0; i < NS; ++i) {
            qa[i] = (r < G) ? ld_ro(qbase + ((int64_t)r * D + 32 * i + 8 * c) * 2)
                            : make_uint4(0, 0, 0, 0);
            if constexpr (TWO_ROWS)
                qb[i] = (r + 8 < G) ? ld_ro(qbase + ((int64_t)(r + 8) * D + 32 * i + 8 * c) * 2)
                                    : make_uint4(0, 0, 0, 0);
        }
    }

    const int nblk = ceil_div_i(w.t_end - w.t_begin, BS);
    const int blk0 = w.t_begin / BS;
    const int32_t* table = p.block_tables + (int64_t)s * p.max_blocks_per_seq + blk0;
    const int64_t tile_elems = (int64_t)BS * D;
    const int64_t block_stride = (int64_t)p.num_kv_heads * tile_elems;
    const char* kbase = reinterpret_cast<const char*>(p.k_cache) + (int64_t)g * tile_elems * 2;
    const char* vbase = reinterpret_cast<const char*>(p.v_cache) + (int64_t)g * tile_elems * 2;
    const float qk = p.qk_scale_log2;

    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
        acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    float m_a = kNegInf, m_b = kNegInf;      // rows r, r + 8
    float l_a = 0.f, l_b = 0.f;

    for (int chunk = 0; warp + chunk * 32 * NW < nblk; ++chunk) {
        const int first = warp + chunk * 32 * NW;
        int my_entry = -1;
        {
            const int i = first + lane * NW;
            if (i < nblk)
                my_entry = __ldg(table + i);
        }
        const int iters = min(32, ceil_div_i(nblk - first, NW));
        for (int it = 0; it < iters; ++it) {
            const int i = first + it * NW;
            const int phys = __shfl_sync(0xffffffffu, my_entry, it);
            if (phys < 0 || (int64_t)phys >= p.num_blocks) {
                if (lane == 0)
                    flag_error(p.dev_err, PKV_DEVERR_BLOCK_ID);
                continue;
            }
            const char* kt = kbase + (int64_t)phys * block_stride * 2;
            const char* vt = vbase + (int64_t)phys * block_stride * 2;
#pragma unroll
            for (int sb = 0; sb < BS / 16; ++sb) {
                const int tb = w.t_begin + i * BS + sb * 16;   // first token of sub-block
                if (tb >= w.t_end)
                    break;
                // loads: K rows (token r, r + 8), V rows (tokens 2c, 2c+1, 2c+8, 2c+9)
                uint4 kv[2][NS];
                uint4 vv[4][NH];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int i2 = 0; i2 < NS; ++i2)
                        kv[nt][i2] = ld_stream(kt + ((int64_t)(sb * 16 + nt * 8 + r) * D +
                                                     32 * i2 + 8 * c) * 2);
#pragma unroll
                for (int tk = 0; tk < 4; ++tk) {
                    const int tok = sb * 16 + 2 * c + (tk & 1) + 8 * (tk >> 1);
#pragma unroll
                    for (int hv = 0; hv < NH; ++hv)
                        vv[tk][hv] = ld_stream(vt + ((int64_t)tok * D + 64 * hv + 8 * r) * 2);
                }

                // S = Q K^T for tokens tb + [0, 8) and tb + [8, 16)
                float sc[2][4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
                    for (int i2 = 0; i2 < NS; ++i2) {
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            uint32_t a[4];
                            a[0] = reg_of(qa[i2], 2 * u);
                            a[2] = reg_of(qa[i2], 2 * u + 1);
                            if constexpr (TWO_ROWS) {
                                a[1] = reg_of(qb[i2], 2 * u);
                                a[3] = reg_of(qb[i2], 2 * u + 1);
                            } else {
                                a[1] = 0u;
                                a[3] = 0u;
                            }
                            mma16816(sc[nt], a, reg_of(kv[nt][i2], 2 * u),
                                     reg_of(kv[nt][i2], 2 * u + 1), kBf16);
                        }
                    }
                }

                // online softmax (base 2) per row; token of sc[nt][e] is
                // tb + nt*8 + 2c + (e & 1), row r for e < 2, row r + 8 otherwise
                float x[2][4];
                float mx_a = kNegInf, mx_b = kNegInf;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const bool ok = tb + nt * 8 + 2 * c + (e & 1) < w.t_end;
                        x[nt][e] = ok ? sc[nt][e] * qk : kNegInf;
                        if (e < 2)
                            mx_a = fmaxf(mx_a, x[nt][e]);
                        else
                            mx_b = fmaxf(mx_b, x[nt][e]);
                    }
                mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
                mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
                const float mn_a = fmaxf(m_a, mx_a);
                const float mn_b = fmaxf(m_b, mx_b);
                const float al_a = exp2f(m_a - mn_a);
                const float al_b = exp2f(m_b - mn_b);
                m_a = mn_a;
                m_b = mn_b;
                l_a *= al_a;
                l_b *= al_b;
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    acc[j][0] *= al_a;
                    acc[j][1] *= al_a;
                    acc[j][2] *= al_b;
                    acc[j][3] *= al_b;
                }
                float pr[2][4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float mref = e < 2 ? mn_a : mn_b;
                        pr[nt][e] = x[nt][e] == kNegInf ? 0.f : exp2f(x[nt][e] - mref);
                        if (e < 2)
                            l_a += pr[nt][e];
                        else
                            l_b += pr[nt][e];
                    }

                // tokens past the context contribute p = 0; clear their V so
                // that whatever bits sit in the unused slots cannot make NaN
#pragma unroll
                for (int tk = 0; tk < 4; ++tk) {
                    const bool ok = tb + 2 * c + (tk & 1) + 8 * (tk >> 1) < w.t_end;
                    if (!ok)
#pragma unroll
                        for (int hv = 0; hv < NH; ++hv)
                            vv[tk][hv] = make_uint4(0, 0, 0, 0);
                }

                // O += P V
                uint32_t ph[4];
                uint32_t pl[4];
                if constexpr (kBf16) {
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) {
                        const int nt = q2 >> 1;
                        const int e0 = (q2 & 1) * 2;
                        const float v0 = pr[nt][e0], v1 = pr[nt][e0 + 1];
                        const uint16_t h0 = round_to<kBF16>(v0), h1 = round_to<kBF16>(v1);
                        const float r0 = v0 - __uint_as_float((uint32_t)h0 << 16);
                        const float r1 = v1 - __uint_as_float((uint32_t)h1 << 16);
                        // fragment order: a0 = row r n-tile 0, a1 = row r+8 n-tile 0,
                        // a2 = row r n-tile 1, a3 = row r+8 n-tile 1
                        ph[q2] = pack2(h0, h1);
                        pl[q2] = pack2(round_to<kBF16>(r0), round_to<kBF16>(r1));
                    }
                } else {
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) {
                        const int nt = q2 >> 1;
                        const int e0 = (q2 & 1) * 2;
                        ph[q2] = pack_f32x2<kF16>(pr[nt][e0], pr[nt][e0 + 1]);
                    }
                }
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const int hv = j / 8;
                    const int e = j % 8;
                    const uint32_t sel = (e & 1) ? 0x7632u : 0x5410u;
                    const uint32_t b0 = __byte_perm(reg_of(vv[0][hv], e >> 1),
                                                    reg_of(vv[1][hv], e >> 1), sel);
                    const uint32_t b1 = __byte_perm(reg_of(vv[2][hv], e >> 1),
                                                    reg_of(vv[3][hv], e >> 1), sel);
                    mma16816(acc[j], ph, b0, b1, kBf16);
                    if constexpr (kBf16)
                        mma16816(acc[j], pl, b0, b1, kBf16);
                }
            }
        }
    }

    // row sums over the four lanes of a row group
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    if (c == 0) {
        sm_m[warp * ROWS + r] = m_a;
        sm_l[warp * ROWS + r] = l_a;
        sm_m[warp * ROWS + r + 8] = m_b;
        sm_l[warp * ROWS + r + 8] = l_b;
    }
    // accumulator of n-tile j, element e: row r (+8 for e >= 2),
    // dim 64*(j/8) + 8*(2c + (e & 1)) + j%8
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int row = r + (e >> 1) * 8;
            const int d = 64 * (j / 8) + 8 * (2 * c + (e & 1)) + (j % 8);
            sm_acc[(warp * ROWS + row) * D + d] = acc[j][e];
        }
    __syncthreads();
    dec::finish_rows<CT, NW, ROWS>(p, w, head0, G, sm_m, sm_l, sm_acc, threadIdx.x,
                                   blockDim.x);
}

// ------------------------------------------------------------------ dispatch

constexpr int kWarps = 4;
// The persistent streaming kernel (decode_stream.cu) serves single-head work
// items; grouped heads use the one-CTA-per-item tensor-core kernel above.
constexpr bool kUseOneCtaPerItem = false;

template <int CT, int QT, int D, int BS>
cudaError_t run_simt(const DecodeParams& p, dim3 grid, cudaStream_t stream)
{
    decode_simt_kernel<CT, QT, D, BS, kWarps><<<grid, kWarps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int CT, int D, int BS>
cudaError_t run_mma(const DecodeParams& p, dim3 grid, cudaStream_t stream)
{
    const size_t smem = sizeof(float) * (2 * kWarps * 16 + kWarps * 16 * D);
    if (p.group > 8) {
        auto kern = decode_mma_kernel<CT, D, BS, kWarps, true>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess)
            return e;
        kern<<<grid, kWarps * 32, smem, stream>>>(p);
    } else {
        auto kern = decode_mma_kernel<CT, D, BS, kWarps, false>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess)
            return e;
        kern<<<grid, kWarps * 32, smem, stream>>>(p);
    }
    return cudaGetLastError();
}

template <int CT, int QT, int D>
cudaError_t simt_bs(const DecodeParams& p, dim3 grid, cudaStream_t st)
{
    switch (p.block_size) {
    case 8:  return run_simt<CT, QT, D, 8>(p, grid, st);
    case 16: return run_simt<CT, QT, D, 16>(p, grid, st);
    case 32: return run_simt<CT, QT, D, 32>(p, grid, st);
    default: return cudaErrorNotSupported;
    }
}

template <int CT, int QT>
cudaError_t simt_d(const DecodeParams& p, dim3 grid, cudaStream_t st)
{
    switch (p.head_dim) {
    case 64:  return simt_bs<CT, QT, 64>(p, grid, st);
    case 128: return simt_bs<CT, QT, 128>(p, grid, st);
    default:  return cudaErrorNotSupported;
    }
}

template <int CT>
cudaError_t mma_shape(const DecodeParams& p, dim3 grid, cudaStream_t st)
{
    if (p.head_dim == 64 && p.block_size == 16) return run_mma<CT, 64, 16>(p, grid, st);
    if (p.head_dim == 64 && p.block_size == 32) return run_mma<CT, 64, 32>(p, grid, st);
    if (p.head_dim == 128 && p.block_size == 16) return run_mma<CT, 128, 16>(p, grid, st);
    if (p.head_dim == 128 && p.block_size == 32) return run_mma<CT, 128, 32>(p, grid, st);
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
    const int64_t ctas = (int64_t)p.max_partitions * p.num_seqs * heads;
    if (ctas <= 0)
        return cudaSuccess;
    if (ctas > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)ctas);
    // one query head per item: the persistent streaming kernel; grouped
    // heads: the one-CTA-per-item tensor-core kernel below
    if (!kUseOneCtaPerItem && !mma)
        return launch_decode_stream(p, false, stream);
    if (mma) {
        return p.cache_dtype == kF16 ? mma_shape<kF16>(p, grid, stream)
                                     : mma_shape<kBF16>(p, grid, stream);
    }
    if (p.cache_dtype == kF16)
        return simt_d<kF16, kF16>(p, grid, stream);
    if (p.cache_dtype == kBF16)
        return simt_d<kBF16, kBF16>(p, grid, stream);
    return p.q_dtype == kF16 ? simt_d<kE4M3, kF16>(p, grid, stream)
                             : simt_d<kE4M3, kBF16>(p, grid, stream);
}

}  // namespace pkv
