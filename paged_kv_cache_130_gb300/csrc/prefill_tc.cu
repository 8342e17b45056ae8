// prefill_tc.cu -- causal prefill attention over the paged cache on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// The prompt phase (「KV Cache从原理到实战」 §2.3): query j of sequence s, at
// position p = context_lens[s] - n_s + j, attends to every cached token t <= p
// (「KV 缓存与分页注意力」 §02).
//
// One CTA = 128 query rows of one (sequence, KV head), rows being (token,
// head) pairs so that the G heads of the KV head share every K/V tile; four
// warps, thread r owns row r and tensor-memory lane r; two CTAs share an SM,
// so one CTA's softmax runs while the other's MMAs do.  Per 64-key tile:
//   * K and V are gathered block by block through the block table with
//     cp.async into 128-byte-swizzled shared-memory panels (64 dims of 64
//     keys per panel; 16-byte chunk c of row r at c ^ (r mod 8)), the layout
//     the tensor core reads: K-major for K, and for V the same bytes read as
//     an MN-major operand.  V_kt and K_{kt+1} load during the softmax of
//     tile kt.
//   * One thread issues S = Q K^T (M = 128, N = 64, K = head_dim) into tensor
//     memory and commits to an mbarrier.
//   * Each thread loads its S row, masks the keys past its position (diagonal
//     tiles only), keeps a running max and sum (fp32, base 2; the max moves
//     only when it grows by more than 2^8, so O in tensor memory is rarely
//     rescaled) and writes P (bf16: a high and a low part, so the weights keep
//     ~16 bits; fp16: one part) into a swizzled P tile.
//   * One thread issues O += P V (M = 128, N = head_dim, K = 64) and the next
//     tile's S.
// The epilogue reads O from tensor memory, divides by the sum and writes the
// rows.  Every mbarrier wait is bounded; on time-out the CTA flags
// PKV_DEVERR_TIMEOUT, skips the rest and still frees its tensor memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kRowsTc = 128;           // query rows per CTA = tensor-memory lanes
constexpr int kKvTc = 64;              // keys per tile
constexpr uint32_t kSpinTc = 1u << 22;
constexpr float kNegInfTc = -__builtin_huge_valf();

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

// Shared-memory matrix descriptor: 128-byte swizzle, version 1 (sm_100 family).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((addr >> 4) & 0x3fff) | ((uint64_t)((lbo >> 4) & 0x3fff) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3fff) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16 with an fp32 accumulator.
template <int CT>
__device__ __forceinline__ uint32_t instr_desc(int m, int n, int b_mn_major)
{
    const uint32_t ab = CT == kBF16 ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)b_mn_major << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                     uint32_t accumulate)
{
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                 " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
                 "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity)
{
    for (uint32_t i = 0; i < kSpinTc; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok)
            return true;
    }
    return false;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
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

__device__ __forceinline__ void bar_expect(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

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

template <int D>
struct TcSmem {
    static constexpr int NP = D / 64;                      // 64-dim panels
    static constexpr int q = 0;                            // [NP][128][128 B]
    static constexpr int k = q + NP * kRowsTc * 128;       // [NP][64][128 B]
    static constexpr int KVT = NP * kKvTc * 128;           // one K or V tile
    static constexpr int v = k + KVT;
    static constexpr int p = v + KVT;                      // [2 parts][128][128 B]
    static constexpr int bytes = p + 2 * kRowsTc * 128;
    static constexpr int alloc = bytes + 1024;             // room to align the base
    static constexpr uint32_t tmem_cols = D == 128 ? 256 : 128;
    static constexpr uint32_t o_col = D == 128 ? 128 : 64; // S at column 0
};

template <int CT, int D, int BS>
__global__ void __launch_bounds__(kRowsTc, 2)
    prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv)
{
    using L = TcSmem<D>;
    constexpr int NCH = D / 8;                 // 16-byte chunks per row
    extern __shared__ unsigned char smem_raw[];
    __shared__ uint32_t tmem_holder;
    __shared__ __align__(8) uint64_t bars[3];  // S done, O done, K/V landed
    __shared__ int abort_flag;
    __shared__ uint32_t bad_rows[2];           // K, V blocks with a bad id (bit per block)

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int G = p.group;
    const int QT = kRowsTc / G;                // new tokens per CTA
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
    auto row_off = [&](int r) -> int64_t {             // element offset of row r in q / out
        return ((int64_t)(cu0 + j0 + r / G) * p.num_heads + g * G + r % G) * D;
    };
    if (bad) {
        if (tid == 0 && j0 == 0 && g == 0)
            flag_error(p.dev_err, PKV_DEVERR_CONTEXT);
        for (int i = tid; i < nrows * (D / 2); i += blockDim.x)
            reinterpret_cast<uint32_t*>(out + row_off(i / (D / 2)))[i % (D / 2)] = 0u;
        return;
    }
    const int pos0 = ctx - n + j0;
    const int kv_end = pos0 + ntok;
    const int nkv = (kv_end + kKvTc - 1) / kKvTc;

    // 1024-byte aligned operand area (the swizzle atoms assume it)
    const uint32_t raw = s_addr(smem_raw);
    unsigned char* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sb = s_addr(base);
    const char* qsrc = reinterpret_cast<const char*>(p.q);
    const int32_t* table = p.block_tables + (int64_t)s * p.max_blocks_per_seq;

    for (int i = tid; i < kRowsTc * NCH; i += blockDim.x) {
        const int r = i / NCH;
        const int c = i % NCH;
        const bool ok = r < nrows;
        cp16z(sb + L::q + panel_off(r, c, kRowsTc), ok ? qsrc + row_off(r) * 2 + c * 16 : qsrc,
              ok);
    }
    // K or V of tile kt -> `which` (L::k or L::v) by TMA, one box per block
    // and 64-dim panel, issued by one thread; returns the bytes to expect.
    // Blocks past kv_end are not loaded (their keys are masked, and the V
    // rows are cleared below); a bad block id is flagged and its rows cleared.
    auto issue_tile = [&](int which, int kt) -> uint32_t {
        const CUtensorMap* map = which == L::k ? &tmk : &tmv;
        uint32_t bytes = 0;
        uint32_t bad = 0;
#pragma unroll
        for (int bi = 0; bi < kKvTc / BS; ++bi) {
            const int tok0 = kt * kKvTc + bi * BS;
            if (tok0 >= kv_end)
                break;
            const int phys = __ldg(table + tok0 / BS);
            if (phys < 0 || (int64_t)phys >= p.num_blocks) {
                bad |= 1u << bi;
                if (which == L::k)
                    flag_error(p.dev_err, PKV_DEVERR_BLOCK_ID);
                continue;
            }
            const int y = (phys * p.num_kv_heads + g) * BS;
#pragma unroll
            for (int pn = 0; pn < D / 64; ++pn)
                tma_box(sb + which + pn * kKvTc * 128 + bi * BS * 128, map, pn * 64, y,
                        s_addr(&bars[2]));
            bytes += (uint32_t)(D / 64) * BS * 128;
        }
        bad_rows[which == L::k ? 0 : 1] = bad;
        return bytes;
    };
    // clear rows [r0, 64) and the rows of bad blocks of a tile (generic
    // stores, made visible to the tensor core by the proxy fence that follows)
    auto clear_rows = [&](int which, int r0, uint32_t bad) {
        for (int i = tid; i < kKvTc * NCH; i += blockDim.x) {
            const int r = i / NCH;
            const int c = i % NCH;
            if (r >= r0 || ((bad >> (r / BS)) & 1u))
                st_v4(base + which + panel_off(r, c, kKvTc), make_uint4(0, 0, 0, 0));
        }
    };
    // Per tile kt (one K and one V buffer; two CTAs share an SM, so one's
    // softmax runs while the other's MMAs do):
    //   wait S_kt; read it; wait P V_{kt-1} (frees V, P and O); TMA V_kt and
    //   K_{kt+1}; softmax, P; then one thread issues O += P_kt V_kt and
    //   S_{kt+1} = Q K_{kt+1}^T.
    asm volatile("cp.async.commit_group;" ::: "memory");                 // Q

    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(s_addr(&bars[0])));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(s_addr(&bars[1])));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(s_addr(&bars[2])));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        abort_flag = 0;
        bar_expect(s_addr(&bars[2]), issue_tile(L::k, 0));
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         s_addr(&tmem_holder)),
                     "r"(L::tmem_cols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();                                                     // barrier init, bad_rows
    if (!bar_wait(s_addr(&bars[2]), 0)) {
        flag_error(p.dev_err, PKV_DEVERR_TIMEOUT);
        abort_flag = 1;
    }
    if (bad_rows[0])
        clear_rows(L::k, kKvTc, bad_rows[0]);
    async_proxy_fence();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_holder;
    const uint32_t lane = (uint32_t)(warp * 32) << 16;     // this warp's tensor-memory lanes
    const uint32_t t_s = tmem + lane;
    const uint32_t t_o = tmem + lane + L::o_col;

    const int row = tid;
    const int pos = pos0 + row / G;            // this row's position
    const float qk = p.qk_scale_log2;
    float m_run = kNegInfTc;                   // running max of the scaled logits
    float l_run = 0.f;
    const uint32_t id_s = instr_desc<CT>(kRowsTc, kKvTc, 0);
    const uint32_t id_o = instr_desc<CT>(kRowsTc, D, 1);
    constexpr int PARTS = CT == kBF16 ? 2 : 1;
    auto issue_s = [&]() {                     // S = Q K^T
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t koff = (uint32_t)(ks & 3) * 32;
            const uint64_t a = smem_desc(sb + L::q + (ks >> 2) * kRowsTc * 128 + koff, 16, 1024);
            const uint64_t bd = smem_desc(sb + L::k + (ks >> 2) * kKvTc * 128 + koff, 16, 1024);
            umma(tmem, a, bd, id_s, ks > 0);
        }
        umma_commit(s_addr(&bars[0]));
    };
    if (tid == 0) {
        tc_fence_after();
        issue_s();
    }

    for (int kt = 0; kt < nkv; ++kt) {
        if (!bar_wait(s_addr(&bars[0]), kt & 1)) {
            flag_error(p.dev_err, PKV_DEVERR_TIMEOUT);
            abort_flag = 1;
        }
        tc_fence_after();
        // this row's 64 raw scores: four loads, one wait
        float x[kKvTc];
#pragma unroll
        for (int c0 = 0; c0 < kKvTc; c0 += 16)
            tmem_ld16(t_s + c0, *reinterpret_cast<uint32_t(*)[16]>(x + c0));
        tmem_wait_ld();
        if (kt > 0) {                          // P V_{kt-1} done: V, P and O are free
            if (!bar_wait(s_addr(&bars[1]), (kt - 1) & 1)) {
                flag_error(p.dev_err, PKV_DEVERR_TIMEOUT);
                abort_flag = 1;
            }
            tc_fence_after();
        }
        if (tid == 0) {                        // S_kt is done with K
            uint32_t bytes = issue_tile(L::v, kt);
            if (kt + 1 < nkv)
                bytes += issue_tile(L::k, kt + 1);
            else
                bad_rows[0] = 0;
            bar_expect(s_addr(&bars[2]), bytes);
        }

        // causal mask only where some key passes some row's position
        if (kt * kKvTc + kKvTc - 1 > pos0) {
#pragma unroll
            for (int j = 0; j < kKvTc; ++j)
                x[j] = kt * kKvTc + j <= pos ? x[j] : kNegInfTc;
        }
        float mx = kNegInfTc;
#pragma unroll
        for (int j = 0; j < kKvTc; ++j)
            mx = fmaxf(mx, x[j]);
        // the running max moves only when a row's max grows by more than 2^8:
        // the weights stay below 256 (exact in fp32) and O is rarely rescaled
        const float m_cand = fmaxf(m_run, mx * qk);
        const bool raise = m_cand > m_run + 8.f;
        const float m_new = raise ? m_cand : m_run;
        const float alpha = raise ? fast_exp2(m_run - m_new) : 1.f;    // 0 on the first tile
        if (kt > 0 && __any_sync(0xffffffffu, raise)) {
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t r32[32];
                tmem_ld16(t_o + c0, *reinterpret_cast<uint32_t(*)[16]>(r32));
                tmem_ld16(t_o + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(r32 + 16));
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    r32[j] = __float_as_uint(__uint_as_float(r32[j]) * alpha);
                tmem_st16(t_o + c0, *reinterpret_cast<uint32_t(*)[16]>(r32));
                tmem_st16(t_o + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(r32 + 16));
            }
            tmem_wait_st();
        }
        m_run = m_new;
        const float neg_m = -m_new;
        float lsum = 0.f;
        unsigned char* prow = base + L::p;
#pragma unroll
        for (int c = 0; c < kKvTc / 8; ++c) {          // 8 keys per 16-byte chunk
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                // exp2(s qk - m); a masked key (-inf) gives 0
                const float p0 = fast_exp2(fmaf(x[8 * c + 2 * e], qk, neg_m));
                const float p1 = fast_exp2(fmaf(x[8 * c + 2 * e + 1], qk, neg_m));
                lsum += p0 + p1;
                hi[e] = pack_rn<CT>(p0, p1);
                if constexpr (CT == kBF16)
                    lo[e] = pack_rn<CT>(p0 - __uint_as_float(hi[e] << 16),
                                        p1 - __uint_as_float(hi[e] & 0xffff0000u));
                else
                    lo[e] = 0u;
            }
            const uint32_t o = panel_off(row, c, kRowsTc);
            st_v4(prow + o, make_uint4(hi[0], hi[1], hi[2], hi[3]));
            if constexpr (CT == kBF16)
                st_v4(prow + kRowsTc * 128 + o, make_uint4(lo[0], lo[1], lo[2], lo[3]));
        }
        l_run = l_run * alpha + lsum;
        if (!bar_wait(s_addr(&bars[2]), (kt + 1) & 1)) {          // V_kt, K_{kt+1}
            flag_error(p.dev_err, PKV_DEVERR_TIMEOUT);
            abort_flag = 1;
        }
        {
            // V rows past kv_end (the last tile) and rows of bad blocks are
            // cleared: P is 0 there, and 0 times stale bits must stay 0
            const int vend = kv_end - kt * kKvTc;
            const uint32_t bad_k = bad_rows[0], bad_v = bad_rows[1];
            if (vend < kKvTc || bad_v)
                clear_rows(L::v, vend < kKvTc ? vend : kKvTc, bad_v);
            if (bad_k)
                clear_rows(L::k, kKvTc, bad_k);
        }
        async_proxy_fence();
        tc_fence_before();
        __syncthreads();
        if (abort_flag)
            break;
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int part = 0; part < PARTS; ++part)
#pragma unroll
                for (int ks = 0; ks < kKvTc / 16; ++ks) {
                    const uint64_t a = smem_desc(sb + L::p + part * kRowsTc * 128 + ks * 32, 16, 1024);
                    // 16 keys further along V's rows; panels of 64 dims are
                    // kKvTc * 128 bytes apart
                    const uint64_t bd = smem_desc(sb + L::v + ks * 16 * 128, kKvTc * 128, 1024);
                    umma(tmem + L::o_col, a, bd, id_o, (kt > 0 || ks > 0 || part > 0) ? 1u : 0u);
                }
            umma_commit(s_addr(&bars[1]));
            if (kt + 1 < nkv)
                issue_s();
        }
    }
    // the last P V
    if (!abort_flag && nkv > 0) {
        if (!bar_wait(s_addr(&bars[1]), (nkv - 1) & 1)) {
            flag_error(p.dev_err, PKV_DEVERR_TIMEOUT);
            abort_flag = 1;
        }
        tc_fence_after();
    }
    __syncthreads();

    // epilogue: O / l for this thread's row
    if (!abort_flag) {
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 16) {
            uint32_t r16[16];
            tmem_ld16(t_o + c0, r16);
            tmem_wait_ld();
            if (row < nrows) {
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    w[e] = pack2(round_to<CT>(__uint_as_float(r16[2 * e]) * inv),
                                 round_to<CT>(__uint_as_float(r16[2 * e + 1]) * inv));
                uint16_t* dst = out + row_off(row) + c0;
                st_v4(dst, make_uint4(w[0], w[1], w[2], w[3]));
                st_v4(dst + 8, make_uint4(w[4], w[5], w[6], w[7]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(L::tmem_cols));
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime.
EncodeTiled encoder()
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
// elements; boxes of 64 elements x BS rows land 128-byte swizzled.
bool cache_map(CUtensorMap* map, const void* cache, int64_t rows, int D, int BS)
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

template <int CT, int D, int BS>
cudaError_t run_prefill_tc(const PrefillParams& p, cudaStream_t stream)
{
    using L = TcSmem<D>;
    auto kern = prefill_tc_kernel<CT, D, BS>;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::alloc);
        if (e != cudaSuccess)
            return e;
        configured[dev] = true;
    }
    const int qt = kRowsTc / p.group;
    const int64_t tiles = (p.max_q_len + qt - 1) / qt;
    const int64_t ctas = tiles * p.num_seqs * p.num_kv_heads;
    if (ctas <= 0)
        return cudaSuccess;
    if (ctas > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    const int64_t rows = p.num_blocks * p.num_kv_heads * BS;
    CUtensorMap tmk, tmv;
    if (!cache_map(&tmk, p.k_cache, rows, D, BS) || !cache_map(&tmv, p.v_cache, rows, D, BS))
        return cudaErrorNotSupported;
    kern<<<(unsigned)ctas, kRowsTc, L::alloc, stream>>>(p, tmk, tmv);
    return cudaGetLastError();
}

template <int CT, int D>
cudaError_t tc_bs(const PrefillParams& p, cudaStream_t st)
{
    switch (p.block_size) {
    case 8: return run_prefill_tc<CT, D, 8>(p, st);
    case 16: return run_prefill_tc<CT, D, 16>(p, st);
    case 32: return run_prefill_tc<CT, D, 32>(p, st);
    default: return cudaErrorNotSupported;
    }
}

template <int CT>
cudaError_t tc_d(const PrefillParams& p, cudaStream_t st)
{
    return p.head_dim == 64 ? tc_bs<CT, 64>(p, st)
                            : (p.head_dim == 128 ? tc_bs<CT, 128>(p, st) : cudaErrorNotSupported);
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillParams& p, cudaStream_t stream)
{
    if (p.num_seqs <= 0 || p.max_q_len <= 0)
        return cudaSuccess;
    if (p.group < 1 || p.group > kRowsTc)
        return cudaErrorNotSupported;
    return p.dtype == kF16 ? tc_d<kF16>(p, stream)
                           : (p.dtype == kBF16 ? tc_d<kBF16>(p, stream) : cudaErrorNotSupported);
}

}  // namespace pkv
