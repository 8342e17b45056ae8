// prefill.cu -- causal prefill attention over the paged cache (tensor cores).
//
// The prompt phase processes all new tokens of a sequence at once
// (「KV Cache从原理到实战」 §2.3): their K/V are appended to the cache first,
// then query j of sequence s, at position p = context_lens[s] - n_s + j,
// attends to every cached token t <= p (「KV 缓存与分页注意力」 §02).  A context
// cached before the new tokens (chunked prefill) is read the same way.
//
// One CTA = 64 query rows of one (sequence, KV head): rows are (token, head)
// pairs, token-major, so the G query heads that share the KV head share every
// K/V tile; 64 / G consecutive new tokens per CTA.  Four warps take 16 rows
// each.  K/V tiles of 64 tokens are gathered block by block through the block
// table with cp.async into a double-buffered, XOR-swizzled shared-memory tile
// (16-byte chunk c of row r at chunk c ^ (r % 8), so that every ldmatrix
// phase touches eight different bank groups).  Per tile and warp:
//   S = Q K^T   mma.sync m16n8k16, A = Q (ldmatrix, kept in registers),
//               B = K (ldmatrix of K[token][dim] rows);
//   causal mask, online softmax (fp32, base 2, rescale only when a row's max
//   rises);
//   O += P V    A = P straight from the S accumulators, B = V (ldmatrix.trans);
//               bf16 P is split into a high and a low part (two MMAs).
// The grid runs the (sequence, KV head) tiles with the most keys first.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kRows = 64;          // query rows per CTA
constexpr int kKv = 64;            // tokens per K/V tile
constexpr int kWarps = 4;
constexpr float kNegInfP = -__builtin_huge_valf();

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// 16-byte global -> shared copy; with valid == false nothing is read and the
// destination is zero-filled (src must still be a mapped address).
__device__ __forceinline__ void cp16(uint32_t dst, const void* src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <bool BF16>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1)
{
    if constexpr (BF16) {
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

// Byte offset of 16-byte chunk c of row r in a swizzled [rows][D] tile.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c)
{
    return (uint32_t)(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

template <int D>
struct PrefillSmem {
    static constexpr int TILE = kKv * D * 2;              // one K or V tile
    static constexpr int q = 0;                           // [kRows][D]
    static constexpr int k = q + kRows * D * 2;           // [2][kKv][D]
    static constexpr int v = k + 2 * TILE;                // [2][kKv][D]
    static constexpr int bytes = v + 2 * TILE;
};

template <int CT, int D, int BS>
__global__ void __launch_bounds__(kWarps * 32, 2) prefill_kernel(const PrefillParams p)
{
    constexpr bool kBf16 = (CT == kBF16);
    constexpr int NC = D / 8;                  // 16-byte chunks per row
    constexpr int NK = D / 16;                 // k-steps of Q K^T
    constexpr int ND = D / 8;                  // output n-tiles
    using L = PrefillSmem<D>;
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t sbase = smem_addr(smem);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int gq = lane >> 2;
    const int t4 = lane & 3;
    const int G = p.group;
    const int QT = kRows / G;                  // new tokens per CTA
    const int ntiles = (p.max_q_len + QT - 1) / QT;
    const int64_t units = (int64_t)p.num_seqs * p.num_kv_heads;
    const int64_t idx = blockIdx.x;
    const int tile = ntiles - 1 - (int)(idx / units);      // heaviest tiles first
    const int s = (int)((idx % units) / p.num_kv_heads);
    const int g = (int)(idx % p.num_kv_heads);

    const int cu0 = __ldg(p.cu_seqlens_q + s);
    const int cu1 = __ldg(p.cu_seqlens_q + s + 1);
    const int n = cu1 - cu0;
    const int j0 = tile * QT;
    if (cu0 < 0 || cu1 < cu0 || cu1 > p.total_q) {
        if (tid == 0 && tile == 0 && g == 0)
            flag_error(p.dev_err, PKV_DEVERR_CONTEXT);
        return;
    }
    if (j0 >= n)
        return;
    const int ctx = __ldg(p.context_lens + s);
    const int ntok = min(QT, n - j0);
    const int nrows = ntok * G;
    const bool bad = ctx < n || ctx > p.max_context_len || n > p.max_q_len ||
                     (ctx + BS - 1) / BS > p.max_blocks_per_seq;
    uint16_t* out = reinterpret_cast<uint16_t*>(p.out);
    auto out_row = [&](int r) -> int64_t {            // element offset of row r
        return ((int64_t)(cu0 + j0 + r / G) * p.num_heads + g * G + r % G) * D;
    };
    if (bad) {
        if (tid == 0 && j0 == 0 && g == 0)
            flag_error(p.dev_err, PKV_DEVERR_CONTEXT);
        for (int i = tid; i < nrows * (D / 2); i += blockDim.x)
            reinterpret_cast<uint32_t*>(out + out_row(i / (D / 2)))[i % (D / 2)] = 0u;
        return;
    }
    const int pos0 = ctx - n + j0;                    // position of token j0
    const int kv_end = pos0 + ntok;                   // keys [0, kv_end)
    const int nkv = (kv_end + kKv - 1) / kKv;

    const char* qsrc = reinterpret_cast<const char*>(p.q);
    const char* kc = reinterpret_cast<const char*>(p.k_cache);
    const char* vc = reinterpret_cast<const char*>(p.v_cache);
    const int32_t* table = p.block_tables + (int64_t)s * p.max_blocks_per_seq;

    // Q rows -> shared memory (zero past nrows)
    for (int i = tid; i < kRows * NC; i += blockDim.x) {
        const int r = i / NC;
        const int c = i % NC;
        const bool ok = r < nrows;
        const char* src = ok ? qsrc + out_row(r) * 2 + c * 16 : qsrc;
        cp16(sbase + L::q + swz<D>(r, c), src, ok);
    }
    // K/V tile kt -> buffer b: 64 keys gathered through the block table; keys
    // past kv_end and bad block ids are zero-filled
    auto load_kv = [&](int kt, int b) {
        for (int i = tid; i < kKv * NC; i += blockDim.x) {
            const int r = i / NC;
            const int c = i % NC;
            const int tok = kt * kKv + r;
            bool ok = tok < kv_end;
            int64_t off = 0;
            if (ok) {
                const int phys = __ldg(table + tok / BS);
                ok = phys >= 0 && (int64_t)phys < p.num_blocks;
                if (!ok && c == 0)
                    flag_error(p.dev_err, PKV_DEVERR_BLOCK_ID);
                off = ((((int64_t)phys * p.num_kv_heads + g) * BS + tok % BS) * D) * 2 + c * 16;
            }
            cp16(sbase + L::k + b * L::TILE + swz<D>(r, c), ok ? kc + off : kc, ok);
            cp16(sbase + L::v + b * L::TILE + swz<D>(r, c), ok ? vc + off : vc, ok);
        }
    };
    load_kv(0, 0);
    cp_commit();

    // per-warp state: rows lo = 16 warp + gq, hi = lo + 8
    const int row_lo = warp * 16 + gq;
    const int pos_lo = pos0 + row_lo / G;
    const int pos_hi = pos0 + (row_lo + 8) / G;
    float o[ND][4];
#pragma unroll
    for (int j = 0; j < ND; ++j)
        o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m_lo = kNegInfP, m_hi = kNegInfP, l_lo = 0.f, l_hi = 0.f;
    uint32_t qa[NK][4];
    const float qk = p.qk_scale_log2;

    for (int kt = 0; kt < nkv; ++kt) {
        if (kt + 1 < nkv)
            load_kv(kt + 1, (kt + 1) & 1);
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        if (kt == 0) {
#pragma unroll
            for (int ks = 0; ks < NK; ++ks) {
                const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                ldsm_x4(qa[ks], sbase + L::q + swz<D>(r, 2 * ks + (lane >> 4)));
            }
        }
        const uint32_t kb_base = sbase + L::k + (kt & 1) * L::TILE;
        const uint32_t vb_base = sbase + L::v + (kt & 1) * L::TILE;

        // S = Q K^T over the tile's 64 keys (8 n-tiles of 8 keys)
        float sc[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
        // k-steps outer: consecutive MMAs update eight independent accumulators
#pragma unroll
        for (int ks = 0; ks < NK; ++ks)
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t kb[4];
                const int r = 16 * np + (lane & 7) + ((lane >> 4) << 3);
                ldsm_x4(kb, kb_base + swz<D>(r, 2 * ks + ((lane >> 3) & 1)));
                mma16816<kBf16>(sc[2 * np], qa[ks], kb[0], kb[1]);
                mma16816<kBf16>(sc[2 * np + 1], qa[ks], kb[2], kb[3]);
            }

        // causal mask and online softmax (base 2)
        const int key0 = kt * kKv + 2 * t4;
        float mx_lo = kNegInfP, mx_hi = kNegInfP;
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = key0 + 8 * j + (e & 1);
                const bool ok = key <= (e < 2 ? pos_lo : pos_hi);
                sc[j][e] = ok ? sc[j][e] * qk : kNegInfP;
                if (e < 2)
                    mx_lo = fmaxf(mx_lo, sc[j][e]);
                else
                    mx_hi = fmaxf(mx_hi, sc[j][e]);
            }
        mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
        mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
        mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
        mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
        const float mn_lo = fmaxf(m_lo, mx_lo);
        const float mn_hi = fmaxf(m_hi, mx_hi);
        if (__any_sync(0xffffffffu, mn_lo > m_lo || mn_hi > m_hi)) {
            const float a_lo = exp2f(m_lo - mn_lo);
            const float a_hi = exp2f(m_hi - mn_hi);
            l_lo *= a_lo;
            l_hi *= a_hi;
#pragma unroll
            for (int j = 0; j < ND; ++j) {
                o[j][0] *= a_lo;
                o[j][1] *= a_lo;
                o[j][2] *= a_hi;
                o[j][3] *= a_hi;
            }
            m_lo = mn_lo;
            m_hi = mn_hi;
        }
        uint32_t ph[4][4];
        uint32_t pl[4][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float pr[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float mref = e < 2 ? m_lo : m_hi;
                pr[e] = sc[j][e] == kNegInfP ? 0.f : exp2f(sc[j][e] - mref);
            }
            l_lo += pr[0] + pr[1];
            l_hi += pr[2] + pr[3];
            // A fragment of k-step j / 2: registers 0, 1 from the even n-tile,
            // 2, 3 from the odd one
            const int kk = j >> 1;
            const int base = (j & 1) * 2;
            if constexpr (kBf16) {
                const uint16_t h0 = round_to<kBF16>(pr[0]), h1 = round_to<kBF16>(pr[1]);
                const uint16_t h2 = round_to<kBF16>(pr[2]), h3 = round_to<kBF16>(pr[3]);
                ph[kk][base] = pack2(h0, h1);
                ph[kk][base + 1] = pack2(h2, h3);
                pl[kk][base] = pack2(round_to<kBF16>(pr[0] - __uint_as_float((uint32_t)h0 << 16)),
                                     round_to<kBF16>(pr[1] - __uint_as_float((uint32_t)h1 << 16)));
                pl[kk][base + 1] =
                    pack2(round_to<kBF16>(pr[2] - __uint_as_float((uint32_t)h2 << 16)),
                          round_to<kBF16>(pr[3] - __uint_as_float((uint32_t)h3 << 16)));
            } else {
                ph[kk][base] = pack2(round_to<kF16>(pr[0]), round_to<kF16>(pr[1]));
                ph[kk][base + 1] = pack2(round_to<kF16>(pr[2]), round_to<kF16>(pr[3]));
                pl[kk][base] = 0u;
                pl[kk][base + 1] = 0u;
            }
        }

        // O += P V (key steps outer, as above)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                uint32_t vb[4];
                const int r = 16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3);
                ldsm_x4_t(vb, vb_base + swz<D>(r, 2 * dp + (lane >> 4)));
                mma16816<kBf16>(o[2 * dp], ph[kk], vb[0], vb[1]);
                mma16816<kBf16>(o[2 * dp + 1], ph[kk], vb[2], vb[3]);
                if constexpr (kBf16) {
                    mma16816<kBf16>(o[2 * dp], pl[kk], vb[0], vb[1]);
                    mma16816<kBf16>(o[2 * dp + 1], pl[kk], vb[2], vb[3]);
                }
            }
        __syncthreads();      // this buffer is refilled two tiles later
    }
    cp_wait<0>();

    // row sums over the four lanes of a row, normalise, write
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
    const float inv_lo = l_lo > 0.f ? 1.f / l_lo : 0.f;
    const float inv_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const int r = row_lo + 8 * hf;
        if (r < nrows) {
            uint16_t* dst = out + out_row(r) + 2 * t4;
            const float inv = hf ? inv_hi : inv_lo;
#pragma unroll
            for (int j = 0; j < ND; ++j)
                *reinterpret_cast<uint32_t*>(dst + 8 * j) =
                    pack2(round_to<CT>(o[j][2 * hf] * inv), round_to<CT>(o[j][2 * hf + 1] * inv));
        }
    }
}

template <int CT, int D, int BS>
cudaError_t run_prefill(const PrefillParams& p, cudaStream_t stream)
{
    using L = PrefillSmem<D>;
    auto kern = prefill_kernel<CT, D, BS>;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::bytes);
        if (e != cudaSuccess)
            return e;
        configured[dev] = true;
    }
    const int qt = kRows / p.group;
    const int64_t tiles = (p.max_q_len + qt - 1) / qt;
    const int64_t ctas = tiles * p.num_seqs * p.num_kv_heads;
    if (ctas <= 0)
        return cudaSuccess;
    if (ctas > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)ctas, kWarps * 32, L::bytes, stream>>>(p);
    return cudaGetLastError();
}

template <int CT, int D>
cudaError_t prefill_bs(const PrefillParams& p, cudaStream_t st)
{
    switch (p.block_size) {
    case 8: return run_prefill<CT, D, 8>(p, st);
    case 16: return run_prefill<CT, D, 16>(p, st);
    case 32: return run_prefill<CT, D, 32>(p, st);
    default: return cudaErrorNotSupported;
    }
}

template <int CT>
cudaError_t prefill_d(const PrefillParams& p, cudaStream_t st)
{
    return p.head_dim == 64 ? prefill_bs<CT, 64>(p, st)
                            : (p.head_dim == 128 ? prefill_bs<CT, 128>(p, st)
                                                 : cudaErrorNotSupported);
}

}  // namespace

bool prefill_shape_supported(int dtype, int head_dim, int block_size, int group)
{
    return (dtype == kF16 || dtype == kBF16) && (head_dim == 64 || head_dim == 128) &&
           (block_size == 8 || block_size == 16 || block_size == 32) && group >= 1 &&
           group <= kRows;
}

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream)
{
    if (!prefill_shape_supported(p.dtype, p.head_dim, p.block_size, p.group))
        return cudaErrorNotSupported;
    if (p.num_seqs <= 0 || p.max_q_len <= 0)
        return cudaSuccess;
    return p.dtype == kF16 ? prefill_d<kF16>(p, stream) : prefill_d<kBF16>(p, stream);
}

}  // namespace pkv
