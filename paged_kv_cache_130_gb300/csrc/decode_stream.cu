// decode_stream.cu -- persistent, warp-specialised decode partition kernel.
//
// The grid holds a few CTAs per SM.  Each CTA walks a static, strided list of
// work items (partition, sequence, head unit).  One producer warp looks up each
// block through the block table (「KV 缓存与分页注意力」 §07 块表) and streams the
// whole (block, KV head) tile of K and of V -- one contiguous run each -- into
// a shared-memory ring with cp.async.bulk, signalling an mbarrier per stage.
// Consumer warps take the ring's stages in turn, keep an online softmax (fp32,
// base 2) and an fp32 P.V accumulator per item, and merge through shared
// memory at the end of each item.  Because the producer runs ahead across item
// boundaries, the dependent loads that start an item (context length, table
// entries) overlap the previous item's stream.
//
// Every wait on an mbarrier is bounded; on time-out the CTA sets
// PKV_DEVERR_TIMEOUT, stops waiting everywhere, lets its in-flight copies land
// and finishes.  There is no other wait in the kernel.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "decode_common.cuh"
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

using dec::ceil_div_i;
using dec::kNegInf;
using dec::PartitionWork;

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
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

// global -> shared bulk copy, completion counted in bytes on `bar`
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(const void* p)
{
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(smem_addr(p)));
    return r;
}

// named barrier over the consumer warps only
__device__ __forceinline__ void consumers_sync(int nthreads)
{
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// Bounded wait for phase `parity` of `bar`.  Returns false when the CTA has
// given up (time-out here or elsewhere); the caller then skips the stage.
constexpr uint32_t kSpinLimit = 1u << 22;

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity,
                                             volatile int* abort_flag, int32_t* dev_err)
{
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*abort_flag)
            return false;
    }
    *abort_flag = 1;
    flag_error(dev_err, PKV_DEVERR_TIMEOUT);
    return false;
}

// ------------------------------------------------------------------ CUDA-core consumer

// One query head against one (block, KV head) tile in shared memory.
// Lane layout: vector j of lane l holds token j*TPI + l/RV, elements
// (l%RV)*EPV .. +EPV (the tile's own byte order: conflict-free 16-byte reads).
template <int CT, int D, int BS>
struct SimtTile {
    static constexpr int C = Elem<CT>::bytes;
    static constexpr int EPV = 16 / C;
    static constexpr int RV = D / EPV;          // lanes per token row
    static constexpr int TPI = 32 / RV;         // tokens per warp-wide read
    static constexpr int NV = BS / TPI;         // vectors per lane per tile
    static constexpr int DUP = RV / NV;         // lanes holding each reduced dot
    static_assert(32 % RV == 0 && BS % TPI == 0 && NV <= RV, "tile shape");

    // state of one item
    float m;
    float l;
    float acc[EPV];

    __device__ __forceinline__ void reset()
    {
        m = kNegInf;
        l = 0.f;
#pragma unroll
        for (int e = 0; e < EPV; ++e)
            acc[e] = 0.f;
    }

    // qf: this lane's EPV query values times scale * log2(e) * k_scale.
    // tok0: token index of this lane's vector 0; t_end: one past the last token.
    __device__ __forceinline__ void consume(const char* sk, const char* sv, const float* qf,
                                            int lane, int tok0, int t_end)
    {
        float x[NV];
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            float kf[EPV];
            unpack_vec<CT>(ld_shared_v4(sk + (j * 32 + lane) * 16), kf);
            float dot = 0.f;
#pragma unroll
            for (int e = 0; e < EPV; ++e)
                dot = fmaf(qf[e], kf[e], dot);
            x[j] = dot;
        }
        // transpose-reduce the NV partial dots over the RV lanes of a row: each
        // round halves the list a lane keeps, so after log2(NV) rounds lane l
        // holds the full dot of token index jsel(l); further rounds finish it.
        int jsel = 0;
#pragma unroll
        for (int half = NV / 2, off = RV / 2; half >= 1; half >>= 1, off >>= 1) {
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int k = 0; k < half; ++k) {
                const float send = upper ? x[k] : x[k + half];
                const float keep = upper ? x[k + half] : x[k];
                x[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
            if (upper)
                jsel += half;
        }
        float dot = x[0];
#pragma unroll
        for (int off = DUP / 2; off >= 1; off >>= 1)
            dot += __shfl_xor_sync(0xffffffffu, dot, off);
        const int my_tok = tok0 + jsel * TPI;
        const float xs = my_tok < t_end ? dot : kNegInf;
        float mx = xs;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m, mx);
        const float alpha = exp2f(m - m_new);
        m = m_new;
        const float p = my_tok < t_end ? exp2f(xs - m_new) : 0.f;
        l = l * alpha + p;
#pragma unroll
        for (int e = 0; e < EPV; ++e)
            acc[e] *= alpha;
        // P.V: the weight of token j sits in lane (row base) + j*DUP
        const int row_base = lane & ~(RV - 1);
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const float pj = __shfl_sync(0xffffffffu, p, row_base + j * DUP);
            if (tok0 + j * TPI < t_end) {
                float vf[EPV];
                unpack_vec<CT>(ld_shared_v4(sv + (j * 32 + lane) * 16), vf);
#pragma unroll
                for (int e = 0; e < EPV; ++e)
                    acc[e] = fmaf(pj, vf[e], acc[e]);
            }
        }
    }

    // Totals over the warp: l over distinct tokens, acc over the lanes of one
    // d-chunk.  Lane l < RV then holds d-chunk l.
    __device__ __forceinline__ void finish_warp()
    {
#pragma unroll
        for (int off = 1; off < 32; off <<= 1)
            l += __shfl_xor_sync(0xffffffffu, l, off);
        l *= 1.0f / DUP;                          // each token counted DUP times
#pragma unroll
        for (int off = RV; off < 32; off <<= 1)
#pragma unroll
            for (int e = 0; e < EPV; ++e)
                acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
    }
};

// ------------------------------------------------------------------ tensor-core consumer

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

__device__ __forceinline__ uint32_t word(const uint4& v, int i)
{
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// All G <= 16 query heads of one KV head against one tile, with
// mma.sync m16n8k16 (fp32 accumulate), per 16-token sub-block:
//   S = Q K^T : rows = query heads (padded to 16), 2 n-tiles of 8 tokens,
//               k-steps over head_dim.  Inside each 32-wide slice head_dim is
//               permuted (thread (r, c) holds dims 32s + 8c + 4u + {0,1},{2,3}
//               for k-step 2s + u) identically for Q and K, so every fragment
//               register comes from one 16-byte read and no dot changes.
//   O += P V : A = P from the S accumulators (rows = heads, k = tokens);
//               output column n of n-tile j is dim 64(j/8) + 8n + j%8, so the
//               B values of one token come from one 16-byte read per 64 dims.
// bf16 P is split into high and low bf16 parts (two MMAs, ~16 bits kept);
// fp16 P is used directly.  Tokens past the context get p = 0 and their V is
// cleared, so unwritten slots cannot reach the sums.
template <int CT, int D, int BS, bool TWO_ROWS, int SK, int SV>
struct MmaTile {
    static constexpr bool kBf16 = (CT == kBF16);
    static constexpr int NS = D / 32;
    static constexpr int NH = D / 64;
    static constexpr int NT = D / 8;
    static_assert(BS % 16 == 0 && D % 64 == 0, "tile shape");

    float acc[NT][4];
    float m_a, m_b, l_a, l_b;        // rows r and r + 8 of this lane

    __device__ __forceinline__ void reset()
    {
#pragma unroll
        for (int j = 0; j < NT; ++j)
            acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
        m_a = m_b = kNegInf;
        l_a = l_b = 0.f;
    }

    __device__ __forceinline__ void consume(const char* sk, const char* sv, const uint4* qa,
                                            const uint4* qb, int lane, int tile_tok0, int t_end,
                                            float qk)
    {
        const int r = lane >> 2;
        const int c = lane & 3;
#pragma unroll
        for (int sb = 0; sb < BS / 16; ++sb) {
            const int tb = tile_tok0 + sb * 16;
            if (tb >= t_end)
                break;
            float sc[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
                for (int i2 = 0; i2 < NS; ++i2) {
                    const uint4 kv = ld_shared_v4(sk + (sb * 16 + nt * 8 + r) * SK + (32 * i2 + 8 * c) * 2);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        uint32_t a[4];
                        a[0] = word(qa[i2], 2 * u);
                        a[2] = word(qa[i2], 2 * u + 1);
                        if constexpr (TWO_ROWS) {
                            a[1] = word(qb[i2], 2 * u);
                            a[3] = word(qb[i2], 2 * u + 1);
                        } else {
                            a[1] = 0u;
                            a[3] = 0u;
                        }
                        mma16816(sc[nt], a, word(kv, 2 * u), word(kv, 2 * u + 1), kBf16);
                    }
                }
            }
            // online softmax (base 2); element e of n-tile nt is token
            // tb + nt*8 + 2c + (e & 1), row r (e < 2) or r + 8
            // rows r + 8 exist only when the group has more than 8 heads
            constexpr int NE = TWO_ROWS ? 4 : 2;
            float x[2][4];
            float mx_a = kNegInf, mx_b = kNegInf;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < NE; ++e) {
                    const bool ok = tb + nt * 8 + 2 * c + (e & 1) < t_end;
                    x[nt][e] = ok ? sc[nt][e] * qk : kNegInf;
                    if (e < 2)
                        mx_a = fmaxf(mx_a, x[nt][e]);
                    else
                        mx_b = fmaxf(mx_b, x[nt][e]);
                }
            mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
            mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
            const float mn_a = fmaxf(m_a, mx_a);
            const float al_a = exp2f(m_a - mn_a);
            m_a = mn_a;
            l_a *= al_a;
            float mn_b = 0.f;
            float al_b = 1.f;
            if constexpr (TWO_ROWS) {
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
                mn_b = fmaxf(m_b, mx_b);
                al_b = exp2f(m_b - mn_b);
                m_b = mn_b;
                l_b *= al_b;
            }
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                acc[j][0] *= al_a;
                acc[j][1] *= al_a;
                if constexpr (TWO_ROWS) {
                    acc[j][2] *= al_b;
                    acc[j][3] *= al_b;
                }
            }
            float pr[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (e >= NE) {
                        pr[nt][e] = 0.f;
                        continue;
                    }
                    const float mref = e < 2 ? mn_a : mn_b;
                    pr[nt][e] = x[nt][e] == kNegInf ? 0.f : exp2f(x[nt][e] - mref);
                    if (e < 2)
                        l_a += pr[nt][e];
                    else
                        l_b += pr[nt][e];
                }
            // P fragments: a0 = row r n-tile 0, a1 = row r+8 n-tile 0,
            // a2 = row r n-tile 1, a3 = row r+8 n-tile 1
            uint32_t ph[4];
            uint32_t pl[4];
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {
                const int nt = q2 >> 1;
                const int e0 = (q2 & 1) * 2;
                const float v0 = pr[nt][e0], v1 = pr[nt][e0 + 1];
                if constexpr (kBf16) {
                    const uint16_t h0 = round_to<kBF16>(v0), h1 = round_to<kBF16>(v1);
                    const float r0 = v0 - __uint_as_float((uint32_t)h0 << 16);
                    const float r1 = v1 - __uint_as_float((uint32_t)h1 << 16);
                    ph[q2] = pack2(h0, h1);
                    pl[q2] = pack2(round_to<kBF16>(r0), round_to<kBF16>(r1));
                } else {
                    ph[q2] = pack2(round_to<kF16>(v0), round_to<kF16>(v1));
                    pl[q2] = 0u;
                }
            }
            // V rows of tokens 2c, 2c+1, 2c+8, 2c+9 (cleared past the context)
            uint4 vv[4][NH];
#pragma unroll
            for (int tk = 0; tk < 4; ++tk) {
                const int tok = 2 * c + (tk & 1) + 8 * (tk >> 1);
                const bool ok = tb + tok < t_end;
#pragma unroll
                for (int hv = 0; hv < NH; ++hv)
                    vv[tk][hv] = ok ? ld_shared_v4(sv + (sb * 16 + tok) * SV + (64 * hv + 8 * r) * 2)
                                    : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int hv = j / 8;
                const int e = j % 8;
                const uint32_t sel = (e & 1) ? 0x7632u : 0x5410u;
                const uint32_t b0 = __byte_perm(word(vv[0][hv], e >> 1), word(vv[1][hv], e >> 1), sel);
                const uint32_t b1 = __byte_perm(word(vv[2][hv], e >> 1), word(vv[3][hv], e >> 1), sel);
                mma16816(acc[j], ph, b0, b1, kBf16);
                if constexpr (kBf16)
                    mma16816(acc[j], pl, b0, b1, kBf16);
            }
        }
    }

    // Row sums over the four lanes of a row group, then this warp's rows
    // into shared memory: sm_m / sm_l [ROWS], sm_acc [ROWS][D] (rows < nrows).
    __device__ __forceinline__ void store_warp(float* sm_m, float* sm_l, float* sm_acc, int lane,
                                               int nrows)
    {
        const int r = lane >> 2;
        const int c = lane & 3;
        l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
        l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
        if (c == 0) {
            if (r < nrows) {
                sm_m[r] = m_a;
                sm_l[r] = l_a;
            }
            if (r + 8 < nrows) {
                sm_m[r + 8] = m_b;
                sm_l[r + 8] = l_b;
            }
        }
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = r + (e >> 1) * 8;
                const int d = 64 * (j / 8) + 8 * (2 * c + (e & 1)) + (j % 8);
                if (row < nrows)
                    sm_acc[row * D + d] = acc[j][e];
            }
    }
};

// Grouped heads, G <= 8, tokens as the MMA rows (no padded rows):
//   S^T = K Q^T : A = K (16 tokens x 16 dims per k-step), B = Q^T (8 heads);
//                 the head_dim permutation inside each 32-wide slice is the
//                 one above, so the K and Q reads are unchanged.
//   O^T += V^T P: A = V^T (16 dims x 16 tokens), B = P (16 tokens x 8 heads).
//                 P leaves the S^T accumulators as (token, head) pairs and is
//                 transposed in registers with movmatrix.  Row r of m-tile j
//                 is dim 8r + j, row r + 8 is dim 64 + 8r + j (head_dim 128)
//                 or 8r + 4 + j (head_dim 64), so a thread's V values of one
//                 token come from one 16-byte read per 64 dims.
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

template <int CT, int D, int BS>
struct GqaTile {
    static constexpr bool kBf16 = (CT == kBF16);
    static constexpr int NS = D / 32;           // 32-wide slices: two k-steps each
    static constexpr int NH = D / 64;           // 16-byte V reads per token
    static constexpr int MT = D / 16;           // m-tiles of O^T
    static_assert(BS % 16 == 0 && (D == 64 || D == 128), "tile shape");

    float acc[MT][4];                           // (dim, head 2c | 2c+1) pairs
    float m0, m1, l0, l1;                       // heads 2c and 2c+1 of this lane

    __device__ __forceinline__ void reset()
    {
#pragma unroll
        for (int j = 0; j < MT; ++j)
            acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
        m0 = m1 = kNegInf;
        l0 = l1 = 0.f;
    }

    // qa: this lane's Q fragment slices of head r (zero past the group)
    __device__ __forceinline__ void consume(const char* sk, const char* sv, const uint4* qa,
                                            int lane, int tile_tok0, int t_end, float qk)
    {
        const int r = lane >> 2;
        const int c = lane & 3;
#pragma unroll
        for (int sb = 0; sb < BS / 16; ++sb) {
            const int tb = tile_tok0 + sb * 16;
            if (tb >= t_end)
                break;
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i2 = 0; i2 < NS; ++i2) {
                const uint4 k0 = ld_shared_v4(sk + ((sb * 16 + r) * D + 32 * i2 + 8 * c) * 2);
                const uint4 k1 = ld_shared_v4(sk + ((sb * 16 + r + 8) * D + 32 * i2 + 8 * c) * 2);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const uint32_t a[4] = {word(k0, 2 * u), word(k1, 2 * u), word(k0, 2 * u + 1),
                                           word(k1, 2 * u + 1)};
                    mma16816(sc, a, word(qa[i2], 2 * u), word(qa[i2], 2 * u + 1), kBf16);
                }
            }
            // sc[0], sc[1]: token tb + r, heads 2c, 2c+1; sc[2], sc[3]: token tb + r + 8
            const bool ok0 = tb + r < t_end;
            const bool ok1 = tb + r + 8 < t_end;
            const float x00 = ok0 ? sc[0] * qk : kNegInf;
            const float x01 = ok0 ? sc[1] * qk : kNegInf;
            const float x10 = ok1 ? sc[2] * qk : kNegInf;
            const float x11 = ok1 ? sc[3] * qk : kNegInf;
            float mx0 = fmaxf(x00, x10);
            float mx1 = fmaxf(x01, x11);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m0, mx0);
            const float mn1 = fmaxf(m1, mx1);
            const float al0 = exp2f(m0 - mn0);
            const float al1 = exp2f(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            const float p00 = ok0 ? exp2f(x00 - mn0) : 0.f;
            const float p01 = ok0 ? exp2f(x01 - mn1) : 0.f;
            const float p10 = ok1 ? exp2f(x10 - mn0) : 0.f;
            const float p11 = ok1 ? exp2f(x11 - mn1) : 0.f;
            l0 = l0 * al0 + p00 + p10;
            l1 = l1 * al1 + p01 + p11;
#pragma unroll
            for (int j = 0; j < MT; ++j) {
                acc[j][0] *= al0;
                acc[j][1] *= al1;
                acc[j][2] *= al0;
                acc[j][3] *= al1;
            }
            // P as the B operand: transpose the (token, head) pairs per 8 tokens
            uint32_t bh0, bh1, bl0 = 0u, bl1 = 0u;
            if constexpr (kBf16) {
                const uint16_t h00 = round_to<kBF16>(p00), h01 = round_to<kBF16>(p01);
                const uint16_t h10 = round_to<kBF16>(p10), h11 = round_to<kBF16>(p11);
                bh0 = transpose8x8(pack2(h00, h01));
                bh1 = transpose8x8(pack2(h10, h11));
                const float r00 = p00 - __uint_as_float((uint32_t)h00 << 16);
                const float r01 = p01 - __uint_as_float((uint32_t)h01 << 16);
                const float r10 = p10 - __uint_as_float((uint32_t)h10 << 16);
                const float r11 = p11 - __uint_as_float((uint32_t)h11 << 16);
                bl0 = transpose8x8(pack2(round_to<kBF16>(r00), round_to<kBF16>(r01)));
                bl1 = transpose8x8(pack2(round_to<kBF16>(r10), round_to<kBF16>(r11)));
            } else {
                bh0 = transpose8x8(pack2(round_to<kF16>(p00), round_to<kF16>(p01)));
                bh1 = transpose8x8(pack2(round_to<kF16>(p10), round_to<kF16>(p11)));
            }
            // V rows of tokens 2c, 2c+1, 2c+8, 2c+9 (cleared past the context)
            uint4 vv[4][NH];
#pragma unroll
            for (int tk = 0; tk < 4; ++tk) {
                const int tok = 2 * c + (tk & 1) + 8 * (tk >> 1);
                const bool ok = tb + tok < t_end;
#pragma unroll
                for (int hv = 0; hv < NH; ++hv)
                    vv[tk][hv] = ok ? ld_shared_v4(sv + ((sb * 16 + tok) * D + 64 * hv + 8 * r) * 2)
                                    : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < MT; ++j) {
                // row r: element j of the first read; row r + 8: element j of the
                // second read (head_dim 128) or element j + 4 of the first
                const int hb = NH == 2 ? 1 : 0;
                const int eb = NH == 2 ? j : j + 4;
                const uint32_t sa = (j & 1) ? 0x7632u : 0x5410u;
                const uint32_t sb2 = (eb & 1) ? 0x7632u : 0x5410u;
                uint32_t a[4];
                a[0] = __byte_perm(word(vv[0][0], j >> 1), word(vv[1][0], j >> 1), sa);
                a[1] = __byte_perm(word(vv[0][hb], eb >> 1), word(vv[1][hb], eb >> 1), sb2);
                a[2] = __byte_perm(word(vv[2][0], j >> 1), word(vv[3][0], j >> 1), sa);
                a[3] = __byte_perm(word(vv[2][hb], eb >> 1), word(vv[3][hb], eb >> 1), sb2);
                mma16816(acc[j], a, bh0, bh1, kBf16);
                if constexpr (kBf16)
                    mma16816(acc[j], a, bl0, bl1, kBf16);
            }
        }
    }

    // Per-head sums over the lanes sharing c, then this warp's rows into
    // shared memory: sm_m / sm_l [8], sm_acc [8][D] (heads < nrows).
    __device__ __forceinline__ void store_warp(float* sm_m, float* sm_l, float* sm_acc, int lane,
                                               int nrows)
    {
        const int r = lane >> 2;
        const int c = lane & 3;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        if (r == 0) {
            if (2 * c < nrows) {
                sm_m[2 * c] = m0;
                sm_l[2 * c] = l0;
            }
            if (2 * c + 1 < nrows) {
                sm_m[2 * c + 1] = m1;
                sm_l[2 * c + 1] = l1;
            }
        }
#pragma unroll
        for (int j = 0; j < MT; ++j) {
            const int d0 = 8 * r + j;
            const int d1 = NH == 2 ? 64 + 8 * r + j : 8 * r + 4 + j;
            if (2 * c < nrows) {
                sm_acc[(2 * c) * D + d0] = acc[j][0];
                sm_acc[(2 * c) * D + d1] = acc[j][2];
            }
            if (2 * c + 1 < nrows) {
                sm_acc[(2 * c + 1) * D + d0] = acc[j][1];
                sm_acc[(2 * c + 1) * D + d1] = acc[j][3];
            }
        }
    }
};

// ------------------------------------------------------------------ the kernel

constexpr int kCtxCache = 512;        // context lengths kept in shared memory
constexpr int kItemQueue = 4;         // work items the producer may publish ahead
constexpr int kSchedSlots = 1024;     // launches that may be in flight at once

// Dynamic work distribution.  Slot k serves one launch: [0] hands out the next
// work item, [1] counts the CTAs that have stopped taking items.  The array is
// zero when the module loads, and the CTA that stops last resets its slot to
// zero, so every launch finds its slot at zero as long as fewer than
// kSchedSlots launches run at the same time.
__device__ unsigned int g_sched[kSchedSlots][2];

// Stage geometry: each (block, KV head) tile lands as one contiguous run, one
// bulk copy for K and one for V (a copy per token row instead would cost the
// copy engine far more than the rows' bank conflicts cost the consumers).
template <int CT, int D, int BS, int MODE>
struct StreamShape {
    static constexpr int ROW = D * Elem<CT>::bytes;           // bytes of one token row
    static constexpr int TILE = BS * ROW;                     // one K (or V) tile in HBM
    static constexpr int SK = ROW;                            // smem stride of K rows
    static constexpr int SV = ROW;                            // smem stride of V rows
    static constexpr int VOFF = BS * SK;                      // V rows start here
    static constexpr int STAGE = ((BS * (SK + SV)) + 127) / 128 * 128;
    // ring bytes: 64 KiB for the CUDA-core consumer; 48 KiB for the grouped-
    // head consumer, whose merge rows and q slots are larger, so that three
    // CTAs still fit on an SM
    static constexpr int NSTG_RAW = (MODE ? 49152 : 65536) / STAGE;
    static constexpr int NSTG = NSTG_RAW < 4 ? 4 : (NSTG_RAW > 16 ? 16 : NSTG_RAW);
};

// Shared-memory layout of one CTA, in bytes from the (128-aligned) base.
template <int CT, int D, int BS, int NC, int MODE, int ROWS>
struct StreamSmem {
    using S = StreamShape<CT, D, BS, MODE>;
    static constexpr int ring = 0;
    static constexpr int full = ring + S::NSTG * S::STAGE;
    static constexpr int empty = full + 8 * S::NSTG;
    static constexpr int iq_full = empty + 8 * S::NSTG;
    static constexpr int iq_empty = iq_full + 8 * kItemQueue;
    static constexpr int items = iq_empty + 8 * kItemQueue;
    static constexpr int cur = items + 4 * kItemQueue;
    static constexpr int flags = cur + 8;
    static constexpr int abort = flags + 4 * S::NSTG;
    static constexpr int ctx = abort + 16;
    static constexpr int QSLOT = ((ROWS * D * 2 + 127) / 128) * 128;   // q rows of one item
    static constexpr int qbuf = ((ctx + 4 * kCtxCache + 127) / 128) * 128;
    static constexpr int merge_m = qbuf + kItemQueue * QSLOT;
    static constexpr int merge_l = merge_m + 4 * NC * ROWS;
    static constexpr int merge_acc = merge_l + 4 * NC * ROWS;
    static constexpr int bytes = merge_acc + 4 * NC * ROWS * D;
};

// MODE 0: one query head per item, CUDA-core consumer.
// MODE 1: one KV head per item (its G <= ROWS query heads), tensor-core consumer.
template <int CT, int QT, int D, int BS, int NC, int MODE, int ROWS>
__global__ void __launch_bounds__((NC + 1) * 32)
    decode_stream_kernel(const DecodeParams p, const int num_items, const int slot)
{
    using Shape = StreamShape<CT, D, BS, MODE>;
    using L = StreamSmem<CT, D, BS, NC, MODE, ROWS>;
    constexpr int TILE = Shape::TILE;
    constexpr int NSTG = Shape::NSTG;
    constexpr int NCT = NC * 32;                      // consumer threads

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ring = smem + L::ring;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L::empty);
    uint64_t* iq_full = reinterpret_cast<uint64_t*>(smem + L::iq_full);
    uint64_t* iq_empty = reinterpret_cast<uint64_t*>(smem + L::iq_empty);
    volatile int* items = reinterpret_cast<volatile int*>(smem + L::items);
    volatile int* cur = reinterpret_cast<volatile int*>(smem + L::cur);
    volatile int* flags = reinterpret_cast<volatile int*>(smem + L::flags);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::abort);
    int* sm_ctx = reinterpret_cast<int*>(smem + L::ctx);
    float* sm_m = reinterpret_cast<float*>(smem + L::merge_m);
    float* sm_l = reinterpret_cast<float*>(smem + L::merge_l);
    float* sm_acc = reinterpret_cast<float*>(smem + L::merge_acc);
    unsigned char* qbuf = smem + L::qbuf;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTG; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < kItemQueue; ++i) {
            mbar_init(&iq_full[i], 1);
            mbar_init(&iq_empty[i], 1);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    const int ncache = min(p.num_seqs, kCtxCache);
    for (int i = threadIdx.x; i < ncache; i += blockDim.x)
        sm_ctx[i] = __ldg(p.context_lens + i);
    __syncthreads();
    pdl_launch_dependents();

    const int U = MODE ? p.num_kv_heads : p.num_heads;
    const int64_t block_stride = (int64_t)p.num_kv_heads * TILE;

    if (warp == NC) {
        // ---------------------------------------------------------- producer
        // Claims items, publishes each non-idle one to the consumers through
        // the item queue, then streams its tiles into the ring.
        uint32_t t = 0;
        uint32_t armed = 0;          // one past the last tile whose copies started
        int published = 0;
        bool stop = false;
        for (;;) {
            int item = 0;
            if (lane == 0)
                item = (int)atomicAdd(&g_sched[slot][0], 1u);
            item = __shfl_sync(0xffffffffu, item, 0);
            const bool last = item >= num_items;
            int u = 0, s = 0, part = 0;
            PartitionWork w{};
            if (!last) {
                u = item % U;
                const int rest = item / U;
                s = rest % p.num_seqs;
                part = rest / p.num_seqs;
                const int ctx = s < ncache ? sm_ctx[s] : __ldg(p.context_lens + s);
                w = dec::locate_ctx(p, s, part, ctx, false);
                if (w.idle)
                    continue;
            }
            // publish the item (or the end marker)
            const int qs = published % kItemQueue;
            if (lane == 0) {
                const bool ok = published < kItemQueue ||
                                wait_bounded(&iq_empty[qs], ((published / kItemQueue) - 1) & 1,
                                             abort_flag, p.dev_err);
                if (ok) {
                    items[qs] = last ? -1 : item;
                    if (last || w.zero_out || w.zero_partial) {
                        mbar_arrive(&iq_full[qs]);
                    } else {
                        // the item's query rows travel with its queue entry
                        const int head0 = MODE ? u * p.group : u;
                        const uint32_t qbytes = (MODE ? p.group : 1) * D * 2;
                        mbar_arrive_expect_tx(&iq_full[qs], qbytes);
                        bulk_load(qbuf + qs * L::QSLOT,
                                  reinterpret_cast<const char*>(p.q) +
                                      ((int64_t)s * p.num_heads + head0) * D * 2,
                                  qbytes, &iq_full[qs]);
                    }
                }
            }
            ++published;
            stop = __shfl_sync(0xffffffffu, *abort_flag, 0) != 0;
            if (last || stop)
                break;
            if (w.zero_out || w.zero_partial)
                continue;                              // the consumers write it
            const int g = MODE ? u : u / p.group;
            const int nblk = ceil_div_i(w.t_end - w.t_begin, BS);
            const int32_t* table =
                p.block_tables + (int64_t)s * p.max_blocks_per_seq + w.t_begin / BS;
            const char* kbase = reinterpret_cast<const char*>(p.k_cache) + (int64_t)g * TILE;
            const char* vbase = reinterpret_cast<const char*>(p.v_cache) + (int64_t)g * TILE;
            for (int c0 = 0; c0 < nblk && !stop; c0 += 32) {
                const int n = min(32, nblk - c0);
                const int entry = lane < n ? __ldg(table + c0 + lane) : -1;
                for (int j = 0; j < n; ++j) {
                    const int phys = __shfl_sync(0xffffffffu, entry, j);
                    const uint32_t stage = t % NSTG;
                    const uint32_t use = t / NSTG;
                    const bool valid = phys >= 0 && (int64_t)phys < p.num_blocks;
                    int ok = 0;
                    if (lane == 0) {
                        ok = use == 0 || wait_bounded(&empty[stage], (use - 1) & 1, abort_flag,
                                                      p.dev_err);
                        if (ok) {
                            flags[stage] = valid ? 1 : 0;
                            if (valid) {
                                mbar_arrive_expect_tx(&full[stage], 2 * TILE);
                            } else {
                                flag_error(p.dev_err, PKV_DEVERR_BLOCK_ID);
                                mbar_arrive(&full[stage]);
                            }
                            armed = t + 1;
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (ok && valid) {
                        unsigned char* dst = ring + stage * Shape::STAGE;
                        const char* ksrc = kbase + (int64_t)phys * block_stride;
                        const char* vsrc = vbase + (int64_t)phys * block_stride;
                        if (lane == 0) {
                            bulk_load(dst, ksrc, TILE, &full[stage]);
                            bulk_load(dst + Shape::VOFF, vsrc, TILE, &full[stage]);
                        }
                    }
                    ++t;
                    stop = __shfl_sync(0xffffffffu, *abort_flag, 0) != 0;
                    if (stop)
                        break;
                }
            }
            if (stop)
                break;
        }
        if (lane == 0) {
            // this CTA takes no more items; the last CTA to get here resets the slot
            __threadfence();
            const unsigned int prev = atomicAdd(&g_sched[slot][1], 1u);
            if (prev == gridDim.x - 1) {
                g_sched[slot][0] = 0u;
                g_sched[slot][1] = 0u;
                __threadfence();
            }
            if (stop) {
                // after a time-out, let the copies already started land (bounded)
                const uint32_t first = armed > (uint32_t)NSTG ? armed - NSTG : 0;
                for (uint32_t tt = first; tt < armed; ++tt)
                    for (uint32_t i = 0; i < kSpinLimit; ++i)
                        if (mbar_try_wait(&full[tt % NSTG], (tt / NSTG) & 1))
                            break;
            }
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    const int ctid = threadIdx.x;                 // 0 .. NCT-1
    const float qk = p.qk_scale_log2;
    uint32_t t = 0;
    for (int n = 0;; ++n) {
        // warp 0 takes the next item from the queue and shares it (two slots,
        // so a slow reader of item n never sees item n+1's value)
        if (warp == 0) {
            const int qs = n % kItemQueue;
            const bool ok = __all_sync(0xffffffffu, wait_bounded(&iq_full[qs], (n / kItemQueue) & 1,
                                                                abort_flag, p.dev_err));
            const int item = ok ? items[qs] : -1;
            __syncwarp();
            if (lane == 0)
                cur[n & 1] = item;
        }
        consumers_sync(NCT);
        const int item = cur[n & 1];
        if (item < 0)
            break;
        const int u = item % U;
        const int rest = item / U;
        const int s = rest % p.num_seqs;
        const int part = rest / p.num_seqs;
        const int ctx = s < ncache ? sm_ctx[s] : __ldg(p.context_lens + s);
        const PartitionWork w = dec::locate_ctx(p, s, part, ctx, ctid == 0);
        const int head0 = MODE ? u * p.group : u;
        const int nrows = MODE ? p.group : 1;
        const int qs = n % kItemQueue;
        const unsigned char* qrow_s = qbuf + qs * L::QSLOT;
        if (w.zero_out || w.zero_partial) {
            if (warp == 0 && lane == 0)
                mbar_arrive(&iq_empty[qs]);
            dec::write_trivial<QT>(p, w, head0, nrows, ctid, NCT);
            continue;
        }
        const int nblk = ceil_div_i(w.t_end - w.t_begin, BS);
        const int k0 = (int)((warp + NC - (int)(t % NC)) % NC);
        // every warp observes the entry's completion itself before reading
        // the q rows the bulk copy wrote (the phase cannot move on before the
        // entry is released below)
        __all_sync(0xffffffffu, wait_bounded(&iq_full[qs], (n / kItemQueue) & 1, abort_flag,
                                             p.dev_err));
        if constexpr (MODE == 0) {
            using T = SimtTile<CT, D, BS>;
            T st;
            st.reset();
            float qf[T::EPV];
            {
                const unsigned char* qrow = qrow_s + (lane % T::RV) * T::EPV * 2;
#pragma unroll
                for (int i = 0; i < T::EPV / 8; ++i)
                    unpack_vec<QT>(ld_shared_v4(qrow + 16 * i), qf + 8 * i);
#pragma unroll
                for (int e = 0; e < T::EPV; ++e)
                    qf[e] *= qk;
            }
            const int tsub = lane / T::RV;
            for (int k = k0; k < nblk; k += NC) {
                const uint32_t tt = t + k;
                const uint32_t stage = tt % NSTG;
                const bool ok = __all_sync(0xffffffffu, wait_bounded(&full[stage], (tt / NSTG) & 1,
                                                                    abort_flag, p.dev_err));
                if (ok && flags[stage]) {
                    const char* sk = reinterpret_cast<const char*>(ring + stage * Shape::STAGE);
                    st.consume(sk, sk + Shape::VOFF, qf, lane, w.t_begin + k * BS + tsub, w.t_end);
                }
                __syncwarp();
                if (ok && lane == 0)
                    mbar_arrive(&empty[stage]);
            }
            st.finish_warp();
            if (lane < T::RV) {
#pragma unroll
                for (int e = 0; e < T::EPV; ++e)
                    sm_acc[warp * D + lane * T::EPV + e] = st.acc[e];
            }
            if (lane == 0) {
                sm_m[warp] = st.m;
                sm_l[warp] = st.l;
            }
        } else if constexpr (ROWS <= 8) {
            using T = GqaTile<CT, D, BS>;
            T st;
            st.reset();
            const int r = lane >> 2;
            const int c = lane & 3;
            uint4 qa[T::NS];
#pragma unroll
            for (int i = 0; i < T::NS; ++i)
                qa[i] = r < nrows ? ld_shared_v4(qrow_s + (r * D + 32 * i + 8 * c) * 2)
                                  : make_uint4(0, 0, 0, 0);
            for (int k = k0; k < nblk; k += NC) {
                const uint32_t tt = t + k;
                const uint32_t stage = tt % NSTG;
                const bool ok = __all_sync(0xffffffffu, wait_bounded(&full[stage], (tt / NSTG) & 1,
                                                                    abort_flag, p.dev_err));
                if (ok && flags[stage]) {
                    const char* sk = reinterpret_cast<const char*>(ring + stage * Shape::STAGE);
                    st.consume(sk, sk + Shape::VOFF, qa, lane, w.t_begin + k * BS, w.t_end, qk);
                }
                __syncwarp();
                if (ok && lane == 0)
                    mbar_arrive(&empty[stage]);
            }
            st.store_warp(sm_m + warp * ROWS, sm_l + warp * ROWS, sm_acc + warp * ROWS * D, lane,
                          nrows);
        } else {
            constexpr bool kTwo = true;
            using T = MmaTile<CT, D, BS, kTwo, Shape::SK, Shape::SV>;
            T st;
            st.reset();
            const int r = lane >> 2;
            const int c = lane & 3;
            uint4 qa[T::NS];
            uint4 qb[kTwo ? T::NS : 1];
            {
#pragma unroll
                for (int i = 0; i < T::NS; ++i) {
                    qa[i] = r < nrows ? ld_shared_v4(qrow_s + (r * D + 32 * i + 8 * c) * 2)
                                      : make_uint4(0, 0, 0, 0);
                    if constexpr (kTwo)
                        qb[i] = r + 8 < nrows
                                    ? ld_shared_v4(qrow_s + ((r + 8) * D + 32 * i + 8 * c) * 2)
                                    : make_uint4(0, 0, 0, 0);
                }
            }
            for (int k = k0; k < nblk; k += NC) {
                const uint32_t tt = t + k;
                const uint32_t stage = tt % NSTG;
                const bool ok = __all_sync(0xffffffffu, wait_bounded(&full[stage], (tt / NSTG) & 1,
                                                                    abort_flag, p.dev_err));
                if (ok && flags[stage]) {
                    const char* sk = reinterpret_cast<const char*>(ring + stage * Shape::STAGE);
                    st.consume(sk, sk + Shape::VOFF, qa, qb, lane, w.t_begin + k * BS, w.t_end, qk);
                }
                __syncwarp();
                if (ok && lane == 0)
                    mbar_arrive(&empty[stage]);
            }
            st.store_warp(sm_m + warp * ROWS, sm_l + warp * ROWS, sm_acc + warp * ROWS * D, lane,
                          nrows);
        }
        t += nblk;
        consumers_sync(NCT);
        // every consumer warp has its q in registers: the queue entry is free
        if (warp == 0 && lane == 0)
            mbar_arrive(&iq_empty[qs]);
        dec::finish_rows<QT, NC, ROWS>(p, w, head0, nrows, sm_m, sm_l, sm_acc, ctid, NCT);
    }
}

std::atomic<unsigned int> g_launch_seq{0};

// Per device and kernel instantiation: the CTAs that fit on the whole GPU,
// worked out (shared-memory opt-in, SM count, occupancy) on the first launch
// and kept, so that later launches cost one cudaLaunchKernel on the host.
constexpr int kMaxDevices = 64;

struct LaunchCache {
    std::mutex mu;
    std::atomic<int> ctas[kMaxDevices];
};

template <typename Kern>
cudaError_t resident_ctas(LaunchCache& cache, Kern kern, int threads, int smem, int* out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    int v = cache.ctas[dev].load(std::memory_order_acquire);
    if (v <= 0) {
        std::lock_guard<std::mutex> lock(cache.mu);
        v = cache.ctas[dev].load(std::memory_order_relaxed);
        if (v <= 0) {
            int sms = 0;
            int per_sm = 0;
            if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          smem)) != cudaSuccess)
                return e;
            if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) !=
                cudaSuccess)
                return e;
            if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads,
                                                                   smem)) != cudaSuccess)
                return e;
            if (per_sm < 1)
                return cudaErrorInvalidConfiguration;
            v = per_sm * sms;
            cache.ctas[dev].store(v, std::memory_order_release);
        }
    }
    *out = v;
    return cudaSuccess;
}

template <int CT, int QT, int D, int BS, int MODE, int ROWS>
cudaError_t run_stream(const DecodeParams& p, cudaStream_t stream)
{
    constexpr int NC = 4;
    using L = StreamSmem<CT, D, BS, NC, MODE, ROWS>;
    auto kern = decode_stream_kernel<CT, QT, D, BS, NC, MODE, ROWS>;
    const int smem = L::bytes;
    static LaunchCache cache;
    int max_ctas = 0;
    cudaError_t e = resident_ctas(cache, kern, (NC + 1) * 32, smem, &max_ctas);
    if (e != cudaSuccess)
        return e;
    const int64_t units = MODE ? p.num_kv_heads : p.num_heads;
    const int64_t items = (int64_t)p.max_partitions * p.num_seqs * units;
    if (items <= 0)
        return cudaSuccess;
    if (items > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    const int64_t grid = items < (int64_t)max_ctas ? items : (int64_t)max_ctas;
    const int slot = (int)(g_launch_seq.fetch_add(1u, std::memory_order_relaxed) % kSchedSlots);
    kern<<<(unsigned)grid, (NC + 1) * 32, smem, stream>>>(p, (int)items, slot);
    return cudaGetLastError();
}

template <int CT, int QT, int D>
cudaError_t stream_simt_bs(const DecodeParams& p, cudaStream_t st)
{
    switch (p.block_size) {
    case 8:  return run_stream<CT, QT, D, 8, 0, 1>(p, st);
    case 16: return run_stream<CT, QT, D, 16, 0, 1>(p, st);
    case 32: return run_stream<CT, QT, D, 32, 0, 1>(p, st);
    default: return cudaErrorNotSupported;
    }
}

template <int CT, int QT>
cudaError_t stream_simt(const DecodeParams& p, cudaStream_t st)
{
    return p.head_dim == 64 ? stream_simt_bs<CT, QT, 64>(p, st)
                            : (p.head_dim == 128 ? stream_simt_bs<CT, QT, 128>(p, st)
                                                 : cudaErrorNotSupported);
}

template <int CT, int D, int BS>
cudaError_t stream_mma_rows(const DecodeParams& p, cudaStream_t st)
{
    return p.group <= 8 ? run_stream<CT, CT, D, BS, 1, 8>(p, st)
                        : run_stream<CT, CT, D, BS, 1, 16>(p, st);
}

template <int CT>
cudaError_t stream_mma(const DecodeParams& p, cudaStream_t st)
{
    if (p.head_dim == 64 && p.block_size == 16) return stream_mma_rows<CT, 64, 16>(p, st);
    if (p.head_dim == 64 && p.block_size == 32) return stream_mma_rows<CT, 64, 32>(p, st);
    if (p.head_dim == 128 && p.block_size == 16) return stream_mma_rows<CT, 128, 16>(p, st);
    if (p.head_dim == 128 && p.block_size == 32) return stream_mma_rows<CT, 128, 32>(p, st);
    return cudaErrorNotSupported;
}

}  // namespace

// Streaming decode partitions; `mma` selects the grouped-head consumer.
cudaError_t launch_decode_stream(const DecodeParams& p, bool mma, cudaStream_t stream)
{
    if (mma) {
        return p.cache_dtype == kF16 ? stream_mma<kF16>(p, stream)
                                     : stream_mma<kBF16>(p, stream);
    }
    if (p.cache_dtype == kF16)
        return stream_simt<kF16, kF16>(p, stream);
    if (p.cache_dtype == kBF16)
        return stream_simt<kBF16, kBF16>(p, stream);
    return p.q_dtype == kF16 ? stream_simt<kE4M3, kF16>(p, stream)
                             : stream_simt<kE4M3, kBF16>(p, stream);
}

}  // namespace pkv
