// prefill_ws.cu -- causal prefill attention over the paged cache, warp
// specialised on the 5th-generation tensor cores.
//
// The prompt phase (「KV Cache从原理到实战」 §2.3): query j of sequence s, at
// position p = context_lens[s] - n_s + j, attends to every cached token t <= p
// (「KV 缓存与分页注意力」 §02).
//
// One CTA = two query tiles (a, b) of 128 rows of one (sequence, KV head); a
// row is a (token, head) pair, so the G heads of the KV head share every K/V
// tile, and both query tiles share each 128-key K/V tile the CTA loads.  Three
// warpgroups; the two softmax groups take 216 registers a thread, the third
// gives its registers up (setmaxnreg) and three of its warps work:
//   * warp 9 (load): walks the block table one slot ahead and gathers, by TMA
//     (one 2-D box per block and 64-dim panel, 128-byte swizzle), slot j =
//     K(j) and V(j-1) into a two-slot shared-memory ring; V blocks past the
//     CTA's last key and blocks with a bad id are zeroed with plain stores,
//     and the V block that holds the context's last token is copied with
//     plain loads and its rows past the context zeroed (they may hold
//     anything, and 0 x NaN would reach the output);
//   * warps 8 and 10 (one issuing thread each, for tiles a and b): per slot j,
//     O_w += P_w(j-1) V(j-1) with P_w read from tensor memory, then
//     S_w(j) = Q_w K(j)^T into the tensor-memory columns P_w occupied; the
//     two threads take turns by slot, each product commits to an mbarrier,
//     and both threads' commits after a slot's last use hand it back to the
//     load warp;
//   * warps 0-3 and 4-7 (softmax of a and of b, thread r = row r = tensor-
//     memory lane r): read S_w, mask the keys past the row's position, keep a
//     running max and sum (fp32, base 2; the max moves only when it grows by
//     more than 2^8, so O is rarely rescaled in tensor memory) and write P_w
//     over S_w (bf16: a high and a low part, so the weights keep ~16 bits;
//     fp16: one part; each 16 keys in their own 16 columns).  While one
//     group's softmax runs, the tensor core works on the other group's
//     products.
// Tensor memory (512 columns): S_a/P_a [0,128), S_b/P_b [128,256),
// O_a [256, 256+D), O_b [256+D, 256+2D).  Every mbarrier wait is bounded; a
// wait that gives up flags PKV_DEVERR_TIMEOUT and makes every role stop, and
// the CTA still waits for its own copies and products and frees its tensor
// memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "tc_common.cuh"

namespace pkv {
namespace {

using namespace tc;

constexpr int kRows = 128;             // rows per query tile = tensor-memory lanes
constexpr int kKeys = 128;             // keys per K/V tile
constexpr int kMmaWarp = 8;            // issues query tile a's products; warp 10 b's
constexpr int kLoadWarp = 9;
constexpr int kThreads = 384;          // three warpgroups: softmax a, softmax b, MMA + load
// registers per thread after the split: 384 x 168 at launch =
// 2 x 128 x kSoftmaxRegs + 128 x kOtherRegs
constexpr int kSoftmaxRegs = 216;
constexpr int kOtherRegs = 72;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kOtherRegs <= kThreads * 168, "register split");
constexpr float kNegInf = -__builtin_huge_valf();

template <int D>
struct WsLayout {
    static constexpr int NP = D / 64;                  // 64-dim panels
    static constexpr int ST = D == 128 ? 2 : 4;        // stages per ring
    static constexpr int QB = NP * kRows * 128;        // one query tile
    static constexpr int KVB = NP * kKeys * 128;       // one K or V tile
    static constexpr int q = 0;                        // [2][NP][128 rows][128 B]
    static constexpr int slot = q + 2 * QB;            // [ST][K, V][NP][128 keys][128 B]
    static constexpr int SLOT = 2 * KVB;               // one slot: K(j), then V(j - 1)
    static constexpr int bytes = slot + ST * SLOT;
    static constexpr int alloc = bytes + 1024;         // room to align the base
    static constexpr uint32_t cols = 512;
};

template <int ST>
struct WsBars {
    uint64_t q_full[2];      // 128 arrivals: the group's Q rows are in shared memory
    uint64_t s_full[2];      // commit: S_w(kt) (and every earlier product of w) done
    uint64_t p_full[2];      // 128 arrivals: P_w(kt) written
    uint64_t o_full[2];      // commit: the last O_w += P_w V done
    uint64_t full[ST];       // slot j landed: K(j) and V(j - 1)
    uint64_t empty[ST];      // one arrival per issuing warp: slot j no longer read
    uint64_t issued[2];      // issuing thread w has queued its products of slot j
    uint64_t drain[2];       // commit: every product issued by warp w done
};

__device__ __forceinline__ bool aborted(const int* flag)
{
    return *reinterpret_cast<const volatile int*>(flag) != 0;
}

__device__ __forceinline__ void set_abort(int* flag, int32_t* dev_err)
{
    *reinterpret_cast<volatile int*>(flag) = 1;
    flag_error(dev_err, PKV_DEVERR_TIMEOUT);
}

// Bounded wait by one thread; gives up early once another role has aborted.
__device__ __forceinline__ bool wait_one(uint32_t bar, uint32_t parity, int* flag,
                                         int32_t* dev_err)
{
    WaitClock clock;
    for (uint32_t i = 0; i < kSpin; ++i) {
        if (try_wait(bar, parity))
            return true;
        if (aborted(flag))
            return false;
        if (clock.expired(i))
            break;
    }
    set_abort(flag, dev_err);
    return false;
}

// The same by a whole warp, with one answer for all its lanes.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, int* flag,
                                          int32_t* dev_err)
{
    bool ok = false;
    WaitClock clock;
    for (uint32_t i = 0; i < kSpin; ++i) {
        if (try_wait(bar, parity)) {
            ok = true;
            break;
        }
        if (aborted(flag) || clock.expired(i))
            break;
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok)
        set_abort(flag, dev_err);
    return ok;
}

template <int CT, int D, int BS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_ws_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv)
{
    using L = WsLayout<D>;
    constexpr int ST = L::ST;
    constexpr int NCH = D / 8;                 // 16-byte chunks per row
    constexpr int NB = kKeys / BS;             // blocks per K/V tile
    constexpr int PARTS = CT == kBF16 ? 2 : 1;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) WsBars<ST> bars;
    __shared__ uint32_t tmem_holder;
    __shared__ int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int G = p.group;
    const int QT = kRows / G;                  // new tokens per query tile
    const int span = 2 * QT;                   // new tokens per CTA
    const int ntiles = (p.max_q_len + span - 1) / span;
    const int64_t units = (int64_t)p.num_seqs * p.num_kv_heads;
    const int64_t idx = blockIdx.x;
    const int tile = ntiles - 1 - (int)(idx / units);      // heaviest tiles first
    const int s = (int)((idx % units) / p.num_kv_heads);
    const int g = (int)(idx % p.num_kv_heads);

    const int cu0 = __ldg(p.cu_seqlens_q + s);
    const int cu1 = __ldg(p.cu_seqlens_q + s + 1);
    const int n = cu1 - cu0;
    const int j0 = tile * span;
    if (cu0 < 0 || cu1 < cu0 || cu1 > p.total_q) {
        if (tid == 0 && tile == 0 && g == 0)
            flag_error(p.dev_err, PKV_DEVERR_CONTEXT);
        return;
    }
    if (j0 >= n)
        return;
    const int ctx = __ldg(p.context_lens + s);
    uint16_t* out = reinterpret_cast<uint16_t*>(p.out);
    auto row_off = [&](int j, int h) -> int64_t {     // element offset of (token j, head h)
        return ((int64_t)(cu0 + j) * p.num_heads + g * G + h) * D;
    };
    if (ctx < n || ctx > p.max_context_len || n > p.max_q_len ||
        (ctx + BS - 1) / BS > p.max_blocks_per_seq) {
        if (tid == 0 && j0 == 0 && g == 0)
            flag_error(p.dev_err, PKV_DEVERR_CONTEXT);
        const int rows = min(span, n - j0) * G;
        for (int i = tid; i < rows * (D / 2); i += blockDim.x) {
            const int r = i / (D / 2);
            reinterpret_cast<uint32_t*>(out + row_off(j0 + r / G, r % G))[i % (D / 2)] = 0u;
        }
        return;
    }
    // the two query tiles: tokens [j0 + w QT, j0 + w QT + ntok_w)
    const int ntok0 = min(QT, n - j0);
    const int ntok1 = max(0, min(QT, n - j0 - QT));
    const int pos00 = ctx - n + j0;            // position of tile a's first token
    const int pos01 = pos00 + QT;
    const int nkv0 = (pos00 + ntok0 + kKeys - 1) / kKeys;
    const int nkv1 = ntok1 > 0 ? (pos01 + ntok1 + kKeys - 1) / kKeys : 0;
    const int nk = max(nkv0, nkv1);            // K/V tiles the CTA loads
    const int kv_end = ntok1 > 0 ? pos01 + ntok1 : pos00 + ntok0;

    const uint32_t raw = s_addr(smem_raw);
    unsigned char* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sb = s_addr(base);

    if (tid == 0) {
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            bar_init(s_addr(&bars.q_full[w]), kRows);
            bar_init(s_addr(&bars.s_full[w]), 1);
            bar_init(s_addr(&bars.p_full[w]), kRows);
            bar_init(s_addr(&bars.o_full[w]), 1);
        }
#pragma unroll
        for (int i = 0; i < ST; ++i) {
            bar_init(s_addr(&bars.full[i]), 1);
            bar_init(s_addr(&bars.empty[i]), ntok1 > 0 ? 2 : 1);
        }
        bar_init(s_addr(&bars.issued[0]), 1);
        bar_init(s_addr(&bars.issued[1]), 1);
        bar_init(s_addr(&bars.drain[0]), 1);
        bar_init(s_addr(&bars.drain[1]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        abort_flag = 0;
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         s_addr(&tmem_holder)),
                     "r"(L::cols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_holder;

    if (warp < 8) {
        // ---------------- softmax of query tile w ----------------
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
        const int w = warp >> 2;
        const int r = tid & (kRows - 1);
        const int ntok = w ? ntok1 : ntok0;
        if (ntok > 0) {
            const int nrows = ntok * G;
            const int jw = j0 + w * QT;
            const int pos0 = w ? pos01 : pos00;
            const int nkv = w ? nkv1 : nkv0;
            {
                const uint32_t qs = sb + L::q + w * L::QB;
                const bool ok = r < nrows;
                const char* src = reinterpret_cast<const char*>(p.q) +
                                  (ok ? row_off(jw + r / G, r % G) * 2 : 0);
#pragma unroll
                for (int c = 0; c < NCH; ++c)
                    cp16z(qs + panel_off(r, c, kRows), src + c * 16, ok);
                asm volatile("cp.async.commit_group;" ::: "memory");
                asm volatile("cp.async.wait_group 0;" ::: "memory");
                async_proxy_fence();
                bar_arrive(s_addr(&bars.q_full[w]));
            }
            const uint32_t lanes = (uint32_t)((warp & 3) * 32) << 16;
            const uint32_t t_s = tmem + lanes + 128u * w;
            const uint32_t t_o = tmem + lanes + 256u + (uint32_t)D * w;
            const int pos = pos0 + r / G;              // this row's position
            const float qk = p.qk_scale_log2;
            float m_run = kNegInf;                     // running max of the scaled logits
            float l_run = 0.f;
            bool alive = true;
            for (int kt = 0; kt < nkv; ++kt) {
                if (!wait_warp(s_addr(&bars.s_full[w]), kt & 1, &abort_flag, p.dev_err)) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                float x[kKeys];
#pragma unroll
                for (int c0 = 0; c0 < kKeys; c0 += 16)
                    tmem_ld16(t_s + c0, *reinterpret_cast<uint32_t(*)[16]>(x + c0));
                tmem_wait_ld();
                // causal mask only where some key passes some row's position
                if (kt * kKeys + kKeys - 1 > pos0) {
#pragma unroll
                    for (int j = 0; j < kKeys; ++j)
                        x[j] = kt * kKeys + j <= pos ? x[j] : kNegInf;
                }
                // row max: eight independent chains of three-input maxima
                float mc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    mc[i] = fmaxf(x[2 * i], x[2 * i + 1]);
#pragma unroll
                for (int j = 16; j < kKeys; j += 16)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        mc[i] = fmax3(mc[i], x[j + 2 * i], x[j + 2 * i + 1]);
                const float mx = fmax3(fmax3(mc[0], mc[1], mc[2]), fmax3(mc[3], mc[4], mc[5]),
                                       fmaxf(mc[6], mc[7]));
                const float m_cand = fmaxf(m_run, mx * qk);
                const bool raise = m_cand > m_run + 8.f;
                const float m_new = raise ? m_cand : m_run;
                const float alpha = raise ? fast_exp2(m_run - m_new) : 1.f;   // 0 on the first tile
                if (kt > 0 && __any_sync(0xffffffffu, raise)) {
                    // O_w += P_w(kt-1) V(kt-1) has completed: the commit behind
                    // S_w(kt) covers every earlier product
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
                }
                m_run = m_new;
                const float2 qk2 = make_float2(qk, qk);
                const float2 nm2 = make_float2(-m_new, -m_new);
                float2 ls[4] = {};                     // four pairs of partial sums
                // P over S, 16 keys at a time in those keys' own 16 columns:
                // 8 columns of high parts, then 8 of low parts, column c of a
                // part holding keys 2c (low half) and 2c + 1
#pragma unroll
                for (int c0 = 0; c0 < kKeys; c0 += 16) {
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        // exp2(s qk - m); a masked key (-inf) gives 0
                        const float2 t = ffma2(make_float2(x[c0 + 2 * e], x[c0 + 2 * e + 1]), qk2, nm2);
                        const float2 pp = make_float2(fast_exp2(t.x), fast_exp2(t.y));
                        ls[e & 3] = fadd2(ls[e & 3], pp);
                        hi[e] = pack_rn<CT>(pp.x, pp.y);
                        if constexpr (CT == kBF16) {
                            const float2 r = fsub2(pp, make_float2(__uint_as_float(hi[e] << 16),
                                                                   __uint_as_float(hi[e] & 0xffff0000u)));
                            lo[e] = pack_rn<CT>(r.x, r.y);
                        } else {
                            lo[e] = 0u;
                        }
                    }
                    tmem_st8(t_s + c0, hi);
                    if constexpr (CT == kBF16)
                        tmem_st8(t_s + c0 + 8, lo);
                }
                const float lsum = ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) +
                                   ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
                tmem_wait_st();
                l_run = l_run * alpha + lsum;
                tc_fence_before();
                bar_arrive(s_addr(&bars.p_full[w]));
            }
            if (alive)
                alive = wait_warp(s_addr(&bars.o_full[w]), 0, &abort_flag, p.dev_err);
            if (alive) {
                // epilogue: O / l for this thread's row
                tc_fence_after();
                const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 16) {
                    uint32_t r16[16];
                    tmem_ld16(t_o + c0, r16);
                    tmem_wait_ld();
                    if (r < nrows) {
                        uint32_t o8[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            o8[e] = pack2(round_to<CT>(__uint_as_float(r16[2 * e]) * inv),
                                          round_to<CT>(__uint_as_float(r16[2 * e + 1]) * inv));
                        uint16_t* dst = out + row_off(jw + r / G, r % G) + c0;
                        st_v4(dst, make_uint4(o8[0], o8[1], o8[2], o8[3]));
                        st_v4(dst + 8, make_uint4(o8[4], o8[5], o8[6], o8[7]));
                    }
                }
            }
        }
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    }
    if ((warp == kMmaWarp || warp == kMmaWarp + 2) && lane == 0 &&
        (warp == kMmaWarp || ntok1 > 0)) {
        // ---------------- tensor-core issue for query tile w (one thread) ----------------
        // Each query tile has its own issuing thread; they take turns by slot
        // (a's P V of slot j, b's, a's of slot j + 1, ...; each thread's S
        // follows its P V and may mix with the other's next P V), so that one
        // tile's softmax runs while the tensor core runs the other tile's
        // products, and each thread's barrier waits overlap the other's
        // queued products.
        const int w = warp == kMmaWarp ? 0 : 1;
        const int nkv = w ? nkv1 : nkv0;
        const uint32_t id_s = instr_desc<CT>(kRows, kKeys, 0);
        const uint32_t id_o = instr_desc<CT>(kRows, D, 1);
        // descriptor halves: every K step only adds (bytes >> 4) to a low half
        constexpr uint32_t hi1k = desc_hi(1024);
        const uint32_t q_lo = desc_lo(sb + L::q + w * L::QB, 16);
        const uint32_t k_lo = desc_lo(sb + L::slot, 16);
        const uint32_t v_lo = desc_lo(sb + L::slot + L::KVB, kKeys * 128);
        const uint32_t s_col = tmem + 128u * w;
        const uint32_t o_col = tmem + 256u + (uint32_t)D * w;
        bool alive = wait_one(s_addr(&bars.q_full[w]), 0, &abort_flag, p.dev_err);
        // slot j: O_w += P_w(j-1) V(j-1), then S_w(j) = Q_w K(j)^T (the S_w
        // columns P_w(j-1) occupied are written after the product read them:
        // one thread's tensor-core operations run in issue order)
        for (int j = 0; alive && j <= nk; ++j) {
            const uint32_t sl = (uint32_t)((j % ST) * L::SLOT >> 4);
            if (!wait_one(s_addr(&bars.full[j % ST]), (j / ST) & 1, &abort_flag, p.dev_err))
                break;
            const bool pv = j > 0 && j <= nkv;
            if (pv && !wait_one(s_addr(&bars.p_full[w]), (j - 1) & 1, &abort_flag, p.dev_err))
                break;
            // the other thread's turn first (its P V of this slot for b, of the
            // slot before for a)
            if (w == 1 ? !wait_one(s_addr(&bars.issued[0]), j & 1, &abort_flag, p.dev_err)
                       : (ntok1 > 0 && j > 0 &&
                          !wait_one(s_addr(&bars.issued[1]), (j - 1) & 1, &abort_flag, p.dev_err)))
                break;
            bool used = false;
            if (pv) {
                tc_fence_after();
                const uint32_t acc0 = j > 1 ? 1u : 0u;
#pragma unroll
                for (int ks = 0; ks < kKeys / 16; ++ks)
#pragma unroll
                    for (int part = 0; part < PARTS; ++part)
                        // 16 keys further along V's rows; 64-dim panels are
                        // kKeys * 128 bytes apart
                        umma_ts_h(o_col, s_col + ks * 16 + part * 8,
                                  v_lo + sl + (uint32_t)(ks * 16 * 128 >> 4), hi1k, id_o,
                                  (ks > 0 || part > 0) ? 1u : acc0);
                if (j == nkv)
                    umma_commit(s_addr(&bars.o_full[w]));
                used = true;
            }
            // the other thread may queue its P V while this one queues S
            bar_arrive(s_addr(&bars.issued[w]));
            if (j < nkv) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (uint32_t)(((ks >> 2) * kRows * 128 + (ks & 3) * 32) >> 4);
                    const uint32_t offk = (uint32_t)(((ks >> 2) * kKeys * 128 + (ks & 3) * 32) >> 4);
                    umma_h(s_col, q_lo + off, hi1k, k_lo + sl + offk, hi1k, id_s, ks > 0 ? 1u : 0u);
                }
                umma_commit(s_addr(&bars.s_full[w]));
                used = true;
            }
            // this thread no longer reads slot j once its products are done
            if (used)
                umma_commit(s_addr(&bars.empty[j % ST]));
            else
                bar_arrive(s_addr(&bars.empty[j % ST]));
        }
        // every product (and every commit's arrival) done before teardown
        umma_commit(s_addr(&bars.drain[w]));
        bar_wait(s_addr(&bars.drain[w]), 0);
    } else if (warp == kLoadWarp) {
        // ---------------- loads (one warp) ----------------
        const int32_t* table = p.block_tables + (int64_t)s * p.max_blocks_per_seq;
        // lane i < NB: physical block i of K/V tile kt; -1 past the CTA's last
        // key, -2 for a bad id
        auto entry = [&](int kt) -> int {
            const int tok = kt * kKeys + lane * BS;
            if (lane >= NB || tok >= kv_end)
                return -1;
            const int phys = __ldg(table + tok / BS);
            if (phys < 0 || (int64_t)phys >= p.num_blocks) {
                flag_error(p.dev_err, PKV_DEVERR_BLOCK_ID);
                return -2;
            }
            return phys;
        };
        int issued = 0;
        // slot j: K(j) (j < nk) and V(j - 1) (j > 0), in one phase of full[j % ST]
        auto load = [&](int j, int ent_k, int ent_v) -> bool {
            const int st = j % ST;
            const uint32_t full = s_addr(&bars.full[st]);
            if (!wait_warp(s_addr(&bars.empty[st]), ((j / ST) & 1) ^ 1, &abort_flag, p.dev_err))
                return false;
            const int tk = j * kKeys + lane * BS;          // first key of K block `lane`
            const int tv = tk - kKeys;                      // first key of V block `lane`
            // by TMA: every block of keys but the V block that holds the
            // context's last token (its rows past the context are not keys)
            const bool tma_k = j < nk && lane < NB && ent_k >= 0;
            const bool tma_v = j > 0 && lane < NB && ent_v >= 0 && tv + BS <= ctx;
            // by plain stores: that block (its keys copied, the other rows
            // zeroed), V blocks past the CTA's last key (zeroed: their weights
            // are 0, and 0 x NaN would not be) and blocks with a bad id
            // (zeroed); K blocks past the last key stay as they are (masked)
            const bool plain_k = j < nk && lane < NB && ent_k == -2;
            const bool plain_v = j > 0 && lane < NB && !tma_v;
            const uint32_t nbox = __popc(__ballot_sync(0xffffffffu, tma_k)) +
                                  __popc(__ballot_sync(0xffffffffu, tma_v));
            if (lane == 0)
                bar_expect_only(full, nbox * (uint32_t)(D / 64) * BS * 128);
            __syncwarp();
            const uint32_t dst = sb + L::slot + st * L::SLOT + lane * BS * 128;
            if (tma_k) {
                const int y = (ent_k * p.num_kv_heads + g) * BS;
#pragma unroll
                for (int pn = 0; pn < D / 64; ++pn)
                    tma_box(dst + pn * kKeys * 128, &tmk, pn * 64, y, full);
            }
            if (tma_v) {
                const int y = (ent_v * p.num_kv_heads + g) * BS;
#pragma unroll
                for (int pn = 0; pn < D / 64; ++pn)
                    tma_box(dst + L::KVB + pn * kKeys * 128, &tmv, pn * 64, y, full);
            }
            uint32_t pm_k = __ballot_sync(0xffffffffu, plain_k);
            uint32_t pm_v = __ballot_sync(0xffffffffu, plain_v);
            if (pm_k | pm_v) {
                while (pm_k | pm_v) {
                    const bool is_v = pm_k == 0;
                    int bl;
                    if (is_v) {
                        bl = __ffs(pm_v) - 1;
                        pm_v &= pm_v - 1;
                    } else {
                        bl = __ffs(pm_k) - 1;
                        pm_k &= pm_k - 1;
                    }
                    const int bent = __shfl_sync(0xffffffffu, is_v ? ent_v : ent_k, bl);
                    // rows that are keys (V: only a block below the last key
                    // that holds the context's last token has some)
                    const int first = (is_v ? j - 1 : j) * kKeys + bl * BS;
                    const int rem = bent >= 0 ? ctx - first : 0;
                    const char* src =
                        reinterpret_cast<const char*>(is_v ? p.v_cache : p.k_cache) +
                        ((int64_t)max(bent, 0) * p.num_kv_heads + g) * BS * D * 2;
                    unsigned char* sdst = base + L::slot + st * L::SLOT + (is_v ? L::KVB : 0);
                    for (int i = lane; i < BS * NCH; i += 32) {
                        const int rr = i / NCH;
                        const int c = i % NCH;
                        const uint4 val = rr < rem ? ld_ro(src + (int64_t)rr * D * 2 + c * 16)
                                                   : make_uint4(0, 0, 0, 0);
                        st_v4(sdst + panel_off(bl * BS + rr, c, kKeys), val);
                    }
                }
                async_proxy_fence();
            }
            __syncwarp();
            if (lane == 0)
                bar_arrive(full);
            ++issued;
            return true;
        };
        int prev = -1;                                     // entries of tile j - 1
        bool alive = true;
        for (int j = 0; alive && j <= nk; ++j) {
            const int cur = j < nk ? entry(j) : -1;
            alive = load(j, cur, prev);
            prev = cur;
        }
        if (!alive) {
            // wait (bounded) for the copies still in flight
            for (int i = max(0, issued - ST); i < issued; ++i)
                bar_wait(s_addr(&bars.full[i % ST]), (i / ST) & 1);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(L::cols));
    }
}

template <int CT, int D, int BS>
cudaError_t run_prefill_ws(const PrefillParams& p, cudaStream_t stream)
{
    using L = WsLayout<D>;
    auto kern = prefill_ws_kernel<CT, D, BS>;
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
    const int span = 2 * (kRows / p.group);
    const int64_t tiles = (p.max_q_len + span - 1) / span;
    const int64_t ctas = tiles * p.num_seqs * p.num_kv_heads;
    if (ctas <= 0)
        return cudaSuccess;
    if (ctas > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    const int64_t rows = p.num_blocks * p.num_kv_heads * BS;
    CUtensorMap tmk, tmv;
    if (!cache_map(&tmk, p.k_cache, rows, D, BS) || !cache_map(&tmv, p.v_cache, rows, D, BS))
        return cudaErrorNotSupported;
    kern<<<(unsigned)ctas, kThreads, L::alloc, stream>>>(p, tmk, tmv);
    return cudaGetLastError();
}

template <int CT, int D>
cudaError_t ws_bs(const PrefillParams& p, cudaStream_t st)
{
    switch (p.block_size) {
    case 8: return run_prefill_ws<CT, D, 8>(p, st);
    case 16: return run_prefill_ws<CT, D, 16>(p, st);
    case 32: return run_prefill_ws<CT, D, 32>(p, st);
    default: return cudaErrorNotSupported;
    }
}

template <int CT>
cudaError_t ws_d(const PrefillParams& p, cudaStream_t st)
{
    return p.head_dim == 64 ? ws_bs<CT, 64>(p, st)
                            : (p.head_dim == 128 ? ws_bs<CT, 128>(p, st) : cudaErrorNotSupported);
}

}  // namespace

cudaError_t launch_prefill_ws(const PrefillParams& p, cudaStream_t stream)
{
    if (p.num_seqs <= 0 || p.max_q_len <= 0)
        return cudaSuccess;
    if (p.group < 1 || p.group > kRows)
        return cudaErrorNotSupported;
    return p.dtype == kF16 ? ws_d<kF16>(p, stream)
                           : (p.dtype == kBF16 ? ws_d<kBF16>(p, stream) : cudaErrorNotSupported);
}

}  // namespace pkv
