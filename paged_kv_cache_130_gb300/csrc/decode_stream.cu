// decode_stream.cu -- persistent, warp-specialised decode partition kernel.
//
// The grid holds as many CTAs as fit on the GPU at once.  Work items are
// (partition, sequence, query head); the CTAs' producer warps claim them from
// a device counter, longest contexts first, one or (for long contexts) a few
// consecutive partitions of one sequence and head at a time.  One producer warp looks up each
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

#include <algorithm>
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

// The same test without suspending: one look at the phase.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
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

// The same with an L2 cache policy for the lines it reads.
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes,
                                               uint64_t* bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
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

// Bounded wait for phase `parity` of `bar`: at most `tries` polls.  Returns
// false when the CTA has given up (time-out here or elsewhere); the caller then
// skips the stage.  A poll is a try_wait, which may suspend the thread for a
// while of the hardware's choosing; under a limit lowered for testing it is a
// test_wait instead, one look, so that a one-poll wait that is not already
// complete always runs out.
constexpr uint32_t kSpinLimit = 1u << 22;

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity,
                                             volatile int* abort_flag, int32_t* dev_err,
                                             uint32_t tries)
{
    const bool look = tries < kSpinLimit;
    WaitClock clock;
    for (uint32_t i = 0; i < tries; ++i) {
        if (look ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if (clock.expired(i))
            break;
    }
    *abort_flag = 1;
    flag_error(dev_err, PKV_DEVERR_TIMEOUT);
    return false;
}

// ------------------------------------------------------------------ CUDA-core consumer

// One query head against one (block, KV head) tile in shared memory.
// Lane layout: vector j of lane l holds token j*TPI + l/RV, elements
// (l%RV)*EPV .. +EPV (the tile's own byte order: conflict-free 16-byte reads).
// Packed fp32 pair arithmetic (two lanes of work per instruction); the
// pairs travel as 64-bit registers inside the asm, so no address is taken.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    float2 r;
    asm("{\n .reg .b64 ra, rb, rc, rd;\n"
        " mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
        " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b)
{
    float2 r;
    asm("{\n .reg .b64 ra, rb, rd;\n"
        " mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
        " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

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
    float2 acc2[EPV / 2];                        // acc[e] = acc2[e / 2].{x, y}

    __device__ __forceinline__ float& acc(int e) { return e & 1 ? acc2[e >> 1].y : acc2[e >> 1].x; }

    __device__ __forceinline__ void reset()
    {
        m = kNegInf;
        l = 0.f;
#pragma unroll
        for (int e = 0; e < EPV / 2; ++e)
            acc2[e] = make_float2(0.f, 0.f);
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
            float2 d2 = make_float2(0.f, 0.f);   // even and odd dims
#pragma unroll
            for (int e = 0; e < EPV; e += 2)
                d2 = ffma2(make_float2(qf[e], qf[e + 1]), make_float2(kf[e], kf[e + 1]), d2);
            x[j] = d2.x + d2.y;
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
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int e = 0; e < EPV / 2; ++e)
            acc2[e] = fmul2(acc2[e], a2);
        // P.V: the weight of token j sits in lane (row base) + j*DUP
        const int row_base = lane & ~(RV - 1);
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const float pj = __shfl_sync(0xffffffffu, p, row_base + j * DUP);
            if (tok0 + j * TPI < t_end) {
                float vf[EPV];
                unpack_vec<CT>(ld_shared_v4(sv + (j * 32 + lane) * 16), vf);
                const float2 p2 = make_float2(pj, pj);
#pragma unroll
                for (int e = 0; e < EPV; e += 2)
                    acc2[e >> 1] = ffma2(p2, make_float2(vf[e], vf[e + 1]), acc2[e >> 1]);
            }
        }
    }

    // Totals over the warp, filed into acc_out[D]: l over distinct tokens
    // (every lane), acc over the 32 / RV lanes that hold one d-chunk.  The
    // acc sums are a transpose reduction: each round over lane bit `off`
    // halves the list a lane keeps (the lane with the bit set keeps the upper
    // half), so after log2(32 / RV) rounds every lane holds D / 32 finished
    // dims and writes them; no sum is computed twice.
    __device__ __forceinline__ void finish_warp(int lane, float* acc_out)
    {
#pragma unroll
        for (int off = 1; off < 32; off <<= 1)
            l += __shfl_xor_sync(0xffffffffu, l, off);
        l *= 1.0f / DUP;                          // each token counted DUP times
        float v[EPV];
#pragma unroll
        for (int e = 0; e < EPV; ++e)
            v[e] = acc(e);
        int first = (lane % RV) * EPV;            // dim of v[0]
#pragma unroll
        for (int off = RV, half = EPV / 2; off < 32; off <<= 1, half >>= 1) {
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int k = 0; k < half; ++k) {
                const float send = upper ? v[k] : v[k + half];
                const float keep = upper ? v[k + half] : v[k];
                v[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
            if (upper)
                first += half;
        }
        constexpr int KEPT = D / 32;
#pragma unroll
        for (int k = 0; k < KEPT; ++k)
            acc_out[first + k] = v[k];
    }
};

// ------------------------------------------------------------------ the kernel

constexpr int kCtxCache = 512;        // context lengths kept in shared memory
constexpr int kSortMax = 128;         // batches up to this size are taken longest first
constexpr int kItemQueue = 4;         // work items the producer may publish ahead
// Work is claimed in units of unit_parts consecutive partitions of one
// (sequence, query head): with contexts of at least kManyParts partitions,
// as many as make up about kUnitTokens tokens (at most kMaxUnitParts), else
// one.  A claim (a device atomic) and the block-table read behind it are
// round trips the producer pays at the start of a unit, not of every
// partition; units much longer than this leave the CTAs uneven at the end.
constexpr int kManyParts = 8;
constexpr int kUnitTokens = 2048;
constexpr int kMaxUnitParts = 4;
// Compact schedule (batches taken longest first, no shared prefixes): units
// where the sequence has no partition left are not handed out at all, and the
// last partitions are handed out one at a time, at least kTailUnits per CTA,
// so that the units the CTAs take last are short.  The schedule is a table of
// at most kMaxSchedEntries (partition block, unit size) entries.
constexpr int kTailUnits = 2;
constexpr int kMaxSchedEntries = 128;
constexpr int kSchedSlots = 1024;     // launches that may be in flight at once

// Dynamic work distribution.  Slot k serves one launch: [0] hands out the next
// work unit after the first gridDim.x (CTA c takes unit c without a claim),
// [1] counts the CTAs that have stopped taking units.  The array is
// zero when the module loads, and the CTA that stops last resets its slot to
// zero, so every launch finds its slot at zero as long as fewer than
// kSchedSlots launches run at the same time.
__device__ unsigned int g_sched[kSchedSlots][2];

// Stage geometry: each (block, KV head) tile lands as one contiguous run, one
// bulk copy for K and one for V, in the tile's own byte order.
template <int CT, int D, int BS>
struct StreamShape {
    static constexpr int TILE = BS * D * Elem<CT>::bytes;     // one K (or V) tile
    static constexpr int VOFF = TILE;                         // V starts here
    static constexpr int STAGE = (2 * TILE + 127) / 128 * 128;
    static constexpr int NSTG_RAW = 65536 / STAGE;           // a 64 KiB ring
    static constexpr int NSTG = NSTG_RAW < 4 ? 4 : (NSTG_RAW > 16 ? 16 : NSTG_RAW);
};

// Shared-memory layout of one CTA, in bytes from the (128-aligned) base.
template <int CT, int D, int BS, int NC>
struct StreamSmem {
    using S = StreamShape<CT, D, BS>;
    static constexpr int ring = 0;
    static constexpr int full = ring + S::NSTG * S::STAGE;
    static constexpr int empty = full + 8 * S::NSTG;
    static constexpr int iq_full = empty + 8 * S::NSTG;
    static constexpr int iq_empty = iq_full + 8 * kItemQueue;
    static constexpr int items = iq_empty + 8 * kItemQueue;
    static constexpr int cur = items + 4 * kItemQueue;
    static constexpr int flags = cur + 8;
    static constexpr int abort = flags + 4 * S::NSTG;
    // the producer's records for the drain at the CTA's end: [0] one past the
    // last ring tile armed, [1] publishes made, [2 + i] whether queue entry i's
    // latest publish started a bulk copy of q
    static constexpr int drain = abort + 16;
    static constexpr int ctx = drain + 4 * (2 + kItemQueue);
    static constexpr int order = ctx + 4 * kCtxCache;
    // the compact schedule: partitions per rank, cumulative units per entry,
    // and [mode, entries, blocks of full units, total units]
    static constexpr int sched_n = order + 4 * kSortMax;
    static constexpr int sched_cum = sched_n + 4 * kSortMax;
    static constexpr int sched_info = sched_cum + 4 * (kMaxSchedEntries + 1);
    static constexpr int QSLOT = ((D * 2 + 127) / 128) * 128;   // q row of one item
    static constexpr int qbuf = ((sched_info + 16 + 127) / 128) * 128;
    static constexpr int merge_m = qbuf + kItemQueue * QSLOT;
    static constexpr int merge_l = merge_m + 4 * NC;
    static constexpr int merge_acc = merge_l + 4 * NC;
    static constexpr int bytes = merge_acc + 4 * NC * D + 1024;
};

// One work item = one (partition, sequence, query head); CUDA-core consumer.
template <int CT, int QT, int D, int BS, int NC>
__global__ void __launch_bounds__((NC + 1) * 32, 3)
    decode_stream_kernel(const DecodeParams p, const int num_items, const int slot,
                         const int unit_parts)
{
    using Shape = StreamShape<CT, D, BS>;
    using L = StreamSmem<CT, D, BS, NC>;
    constexpr int TILE = Shape::TILE;
    constexpr int NSTG = Shape::NSTG;
    constexpr int NCT = NC * 32;                      // consumer threads
    // Tile t goes to consumer warp t % NC and to stage t % NSTG, and the waits
    // on a stage's mbarrier tell its phases apart by parity only.  With NSTG a
    // multiple of NC, tiles t and t + NSTG (consecutive uses of one stage) go
    // to the same warp, which waits for t + NSTG only after consuming t; with
    // any other ring size another warp could wait for t + NSTG before t's copy
    // has landed and take that earlier phase for its own.
    static_assert(NSTG % NC == 0, "ring stages must be a multiple of the consumer warps");

    // the ring starts on a 1024-byte boundary (the layout's last 1024 bytes
    // are the room for it): measured 4 % faster on the E4M3 layer than the
    // base's own alignment
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char* smem =
        smem_raw + (((smem_addr(smem_raw) + 1023u) & ~1023u) - smem_addr(smem_raw));
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
    int* sm_order = reinterpret_cast<int*>(smem + L::order);
    int* sched_n = reinterpret_cast<int*>(smem + L::sched_n);
    int* sched_cum = reinterpret_cast<int*>(smem + L::sched_cum);
    int* sched_info = reinterpret_cast<int*>(smem + L::sched_info);
    float* sm_m = reinterpret_cast<float*>(smem + L::merge_m);
    float* sm_l = reinterpret_cast<float*>(smem + L::merge_l);
    float* sm_acc = reinterpret_cast<float*>(smem + L::merge_acc);
    volatile int* drain = reinterpret_cast<volatile int*>(smem + L::drain);
    unsigned char* qbuf = smem + L::qbuf;
    // polls per wait on the ring and the item queue (a test may lower it to
    // make a wait run out); the drain at the end always has the full limit
    const uint32_t tries = p.wait_tries ? p.wait_tries : kSpinLimit;

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
        for (int i = 0; i < 2 + kItemQueue; ++i)
            drain[i] = 0;
        mbar_init_fence();
    }
    // launched with programmatic dependent launch after whatever the stream
    // ran before: nothing is read before that work is complete (with a
    // shared-prefix kernel before it, see wait_prior, the wait comes at the
    // end instead)
    if (!p.wait_prior)
        pdl_wait_primary();
    const int U = p.num_heads;
    const int ncache = min(p.num_seqs, kCtxCache);
    for (int i = threadIdx.x; i < ncache; i += blockDim.x)
        sm_ctx[i] = __ldg(p.context_lens + i);
    __syncthreads();
    // Longest first: every CTA ranks the sequences by descending context
    // length (ties by index) and walks work items in that order, so that the
    // dynamic scheduler hands out the largest items first and the last ones
    // to finish are short.
    const bool sorted = p.num_seqs <= kSortMax;
    if (sorted) {
        for (int i = threadIdx.x; i < p.num_seqs; i += blockDim.x) {
            const int ci = sm_ctx[i];
            int rank = 0;
            for (int j = 0; j < p.num_seqs; ++j) {
                const int cj = sm_ctx[j];
                rank += (cj > ci) || (cj == ci && j < i);
            }
            sm_order[rank] = i;
        }
    }
    // The compact schedule, the same in every CTA.  Units go out in the order
    // (entry, rank, head); entry j < blocks1 is partition block j (unit_parts
    // partitions from j * unit_parts), each later one a single partition,
    // and an entry holds only the ranks that have a partition there (with
    // the ranks ordered longest first these are a prefix of the ranks).
    if (threadIdx.x == 0)
        sched_info[0] = 0;
    const bool try_compact = sorted && unit_parts > 1 &&
                             (p.grp_begin == nullptr || p.num_groups <= 0);
    if (try_compact) {
        __syncthreads();                                   // sm_order complete
        for (int i = threadIdx.x; i < p.num_seqs; i += blockDim.x) {
            // partitions of rank i's work, as locate_ctx walks them
            const dec::Split sp = dec::split_context(sm_ctx[sm_order[i]], 0, p.max_context_len,
                                                     p.partition_size, p.prefix_partition);
            sched_n[i] = sp.npart <= 1 ? 1 : min(sp.npart, p.grid_partitions);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            const int ns = p.num_seqs;
            bool ok = true;
            for (int i = 1; i < ns; ++i)
                ok = ok && sched_n[i] <= sched_n[i - 1];
            const int maxp = sched_n[0];
            // a table of more than kMaxSchedEntries entries is certain past
            // this point; the scan below then is not made at all
            ok = ok && maxp <= kMaxSchedEntries * unit_parts;
            // the first partition of the single-partition tail: the largest
            // multiple of unit_parts after which at least kTailUnits units a
            // CTA remain (0: every unit a single partition)
            int q2 = 0;
            {
                int r = 0;
                int64_t after = 0;
                for (int q = maxp - 1; q >= 0 && ok; --q) {
                    while (r < ns && sched_n[r] > q)
                        ++r;
                    after += (int64_t)r * U;
                    if (q % unit_parts == 0 && after >= (int64_t)kTailUnits * gridDim.x) {
                        q2 = q;
                        break;
                    }
                }
            }
            const int blocks1 = q2 / unit_parts;
            const int entries = blocks1 + (maxp - q2);
            ok = ok && entries <= kMaxSchedEntries;
            if (ok) {
                int r = ns;
                int64_t cum = 0;
                sched_cum[0] = 0;
                for (int j = 0; j < entries && ok; ++j) {
                    const int q0 = j < blocks1 ? j * unit_parts : q2 + (j - blocks1);
                    while (r > 0 && sched_n[r - 1] <= q0)
                        --r;
                    cum += (int64_t)r * U;
                    ok = cum <= 0x7fffffffLL;
                    sched_cum[j + 1] = (int)cum;
                }
                if (ok) {
                    sched_info[1] = entries;
                    sched_info[2] = blocks1;
                    sched_info[3] = (int)cum;
                    sched_info[0] = 1;
                }
            }
        }
    }
    __syncthreads();
    pdl_launch_dependents();
    const bool compact = sched_info[0] != 0;
    const int total_units = compact ? sched_info[3] : num_items;

    const int64_t block_stride = (int64_t)p.num_kv_heads * TILE;

    // -------------------------------------------------------------- consumers
    // (a lambda, so that the producer and the consumers meet again at the end)
    auto consumer_loop = [&]() {
        const int ctid = threadIdx.x;                 // 0 .. NCT-1
        const float qk = p.qk_scale_log2;
        uint32_t t = 0;
        for (int n = 0;; ++n) {
            // warp 0 takes the next item from the queue and shares it (two slots,
            // so a slow reader of item n never sees item n+1's value)
            if (warp == 0) {
                const int qs = n % kItemQueue;
                const bool ok = __all_sync(
                    0xffffffffu, wait_bounded(&iq_full[qs], (n / kItemQueue) & 1, abort_flag,
                                              p.dev_err, tries));
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
            const int s = sorted ? sm_order[rest % p.num_seqs] : rest % p.num_seqs;
            const int part = rest / p.num_seqs;
            const int ctx = s < ncache ? sm_ctx[s] : __ldg(p.context_lens + s);
            const PartitionWork w = dec::locate_ctx(p, s, part, ctx, ctid == 0);
            const int head0 = u;
            const int nrows = 1;
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
                                                 p.dev_err, tries));
            {
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
                    const bool ok = __all_sync(
                        0xffffffffu, wait_bounded(&full[stage], (tt / NSTG) & 1, abort_flag,
                                                  p.dev_err, tries));
                    if (ok && flags[stage]) {
                        const char* sk =
                            reinterpret_cast<const char*>(ring + stage * Shape::STAGE);
                        st.consume(sk, sk + Shape::VOFF, qf, lane, w.t_begin + k * BS + tsub,
                                   w.t_end);
                    }
                    __syncwarp();
                    if (ok && lane == 0)
                        mbar_arrive(&empty[stage]);
                }
                // filed by block residue k0, not by warp: the merge then adds the
                // same partial sums in the same order whichever warp held a
                // residue (that depends on the items the CTA took before), so a
                // result is the same from run to run, bit for bit
                st.finish_warp(lane, sm_acc + k0 * D);
                if (lane == 0) {
                    sm_m[k0] = st.m;
                    sm_l[k0] = st.l;
                }
            }
            t += nblk;
            consumers_sync(NCT);
            // every consumer warp has its q in registers: the queue entry is
            // free -- unless a wait gave up (a warp whose wait on the entry
            // failed raised the abort flag before this barrier): then the q
            // copy may still be in flight, and the entry stays taken so that
            // no new copy is started into it
            if (warp == 0 && lane == 0 && !*abort_flag)
                mbar_arrive(&iq_empty[qs]);
            dec::finish_rows<QT, NC, 1>(p, w, head0, nrows, sm_m, sm_l, sm_acc, ctid, NCT);
        }
    };

    if (warp == NC) {
        // ---------------------------------------------------------- producer
        // Claims items, publishes each non-idle one to the consumers through
        // the item queue, then streams its tiles into the ring.
        uint32_t t = 0;
        uint32_t armed = 0;          // one past the last tile whose copies started
        // K/V tiles are read once per call: first out of L2
        const uint64_t kv_policy = l2_evict_first_policy();
        int published = 0;
        bool stop = false;
        for (bool first = true;; first = false) {
            // one claim hands out a unit: unit_parts consecutive partitions
            // of one (sequence, query head), streamed back to back so that
            // the claim's and the block table's round trips are paid once.
            // A CTA's first unit is its own index (no round trip before its
            // first table read); the counter hands out the rest from
            // gridDim.x on.
            int unit = 0;
            if (first) {
                unit = (int)blockIdx.x;
            } else if (lane == 0) {
                unit = (int)(atomicAdd(&g_sched[slot][0], 1u) + gridDim.x);
                // the counter serves total_units - gridDim.x units and one
                // failed claim per CTA, so unit < total_units + gridDim.x: a
                // higher one means another launch shares the slot
                if ((unsigned)unit >= (unsigned)total_units + gridDim.x)
                    flag_error(p.dev_err, PKV_DEVERR_SCHED);
            }
            unit = __shfl_sync(0xffffffffu, unit, 0);
            const bool last = unit >= total_units;
            // the unit's (rank, head, first partition, partitions)
            int u_rank = 0, u_head = 0, u_q0 = 0, u_parts = unit_parts;
            if (!last && compact) {
                int lo = 0;
                int hi = sched_info[1];          // the entry j with cum[j] <= unit < cum[j + 1]
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (sched_cum[mid] <= unit)
                        lo = mid;
                    else
                        hi = mid;
                }
                const int local = unit - sched_cum[lo];
                u_rank = local / U;
                u_head = local % U;
                const int blocks1 = sched_info[2];
                u_q0 = lo < blocks1 ? lo * unit_parts : blocks1 * unit_parts + (lo - blocks1);
                u_parts = lo < blocks1 ? unit_parts : 1;
            } else if (!last) {
                u_head = unit % U;
                u_rank = (unit / U) % p.num_seqs;
                u_q0 = (unit / U / p.num_seqs) * unit_parts;
            }
            for (int sub = 0; sub < (last ? 1 : u_parts); ++sub) {
                int item = -1;
                int u = 0, s = 0;
                PartitionWork w{};
                if (!last) {
                    u = u_head;
                    const int rank = u_rank;
                    const int part = u_q0 + sub;
                    if (part >= p.grid_partitions)
                        break;
                    s = sorted ? sm_order[rank] : rank;
                    const int ctx = s < ncache ? sm_ctx[s] : __ldg(p.context_lens + s);
                    w = dec::locate_ctx(p, s, part, ctx, false);
                    if (w.idle)
                        break;                          // and so is every later part
                    item = (part * p.num_seqs + rank) * U + u;
                }
                // publish the item (or the end marker)
                const int qs = published % kItemQueue;
                if (lane == 0) {
                    const bool ok = published < kItemQueue ||
                                    wait_bounded(&iq_empty[qs], ((published / kItemQueue) - 1) & 1,
                                                 abort_flag, p.dev_err, tries);
                    if (ok) {
                        items[qs] = last ? -1 : item;
                        drain[1] = published + 1;
                        const bool copy_q = !(last || w.zero_out || w.zero_partial);
                        drain[2 + qs] = copy_q ? 1 : 0;
                        if (!copy_q) {
                            mbar_arrive(&iq_full[qs]);
                        } else {
                            // the item's query rows travel with its queue entry
                            const int head0 = u;
                            const uint32_t qbytes = D * 2;
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
                const int g = u / p.group;
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
                                                          p.dev_err, tries);
                            if (ok) {
                                flags[stage] = valid ? 1 : 0;
                                if (valid) {
                                    mbar_arrive_expect_tx(&full[stage], 2 * TILE);
                                } else {
                                    flag_error(p.dev_err, PKV_DEVERR_BLOCK_ID);
                                    mbar_arrive(&full[stage]);
                                }
                                armed = t + 1;
                                drain[0] = (int)armed;
                            }
                        }
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        if (ok && valid) {
                            unsigned char* dst = ring + stage * Shape::STAGE;
                            const char* ksrc = kbase + (int64_t)phys * block_stride;
                            const char* vsrc = vbase + (int64_t)phys * block_stride;
                            if (lane == 0) {
                                bulk_load_hint(dst, ksrc, TILE, &full[stage], kv_policy);
                                bulk_load_hint(dst + Shape::VOFF, vsrc, TILE, &full[stage],
                                               kv_policy);
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
            if (last || stop)
                break;
        }
        if (lane == 0) {
            // this CTA takes no more items; the last CTA to get here resets the slot
            __threadfence();
            const unsigned int prev = atomicAdd(&g_sched[slot][1], 1u);
            if (prev >= gridDim.x)
                flag_error(p.dev_err, PKV_DEVERR_SCHED);   // another launch shares the slot
            if (prev == gridDim.x - 1) {
                g_sched[slot][0] = 0u;
                g_sched[slot][1] = 0u;
                __threadfence();
            }
        }
    } else {
        consumer_loop();
    }
    // Every copy this CTA started lands before it exits.  In a run without a
    // time-out the consumers waited for each one already; after one, the
    // copies still in flight are the last NSTG ring tiles armed and the q rows
    // of the last kItemQueue published items (the producer's records are
    // final once every warp has reached this barrier).  These waits keep the
    // full limit whatever the test setting.
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        const uint32_t armed_all = (uint32_t)drain[0];
        const uint32_t first = armed_all > (uint32_t)NSTG ? armed_all - NSTG : 0;
        for (uint32_t tt = first; tt < armed_all; ++tt) {
            WaitClock clock;
            for (uint32_t i = 0; i < kSpinLimit; ++i)
                if (mbar_try_wait(&full[tt % NSTG], (tt / NSTG) & 1) || clock.expired(i))
                    break;
        }
        const int pub = drain[1];
        for (int n = pub > kItemQueue ? pub - kItemQueue : 0; n < pub; ++n) {
            if (!drain[2 + n % kItemQueue])
                continue;
            WaitClock clock;
            for (uint32_t i = 0; i < kSpinLimit; ++i)
                if (mbar_try_wait(&iq_full[n % kItemQueue], (n / kItemQueue) & 1) ||
                    clock.expired(i))
                    break;
        }
    }
    if (p.wait_prior && threadIdx.x == 0)
        pdl_wait_primary();
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

template <int CT, int QT, int D, int BS>
cudaError_t run_stream(const DecodeParams& p, cudaStream_t stream)
{
    constexpr int NC = 4;
    using L = StreamSmem<CT, D, BS, NC>;
    auto kern = decode_stream_kernel<CT, QT, D, BS, NC>;
    const int smem = L::bytes;
    static LaunchCache cache;
    int max_ctas = 0;
    cudaError_t e = resident_ctas(cache, kern, (NC + 1) * 32, smem, &max_ctas);
    if (e != cudaSuccess)
        return e;
    const int64_t units = p.num_heads;
    // units of unit_parts consecutive partitions claimed at once
    int unit_parts = 1;
    if (p.grid_partitions >= kManyParts && p.partition_size > 0)
        unit_parts = std::max(1, std::min(kMaxUnitParts, kUnitTokens / p.partition_size));
    const int64_t items =
        (int64_t)((p.grid_partitions + unit_parts - 1) / unit_parts) * p.num_seqs * units;
    if (items <= 0)
        return cudaSuccess;
    // the ids of single partitions must fit an int as well
    if ((int64_t)p.grid_partitions * p.num_seqs * units > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    const int64_t grid = items < (int64_t)max_ctas ? items : (int64_t)max_ctas;
    const int slot = (int)(g_launch_seq.fetch_add(1u, std::memory_order_relaxed) % kSchedSlots);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((NC + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, (int)items, slot, unit_parts);
}

template <int CT, int QT, int D>
cudaError_t stream_simt_bs(const DecodeParams& p, cudaStream_t st)
{
    switch (p.block_size) {
    case 8:  return run_stream<CT, QT, D, 8>(p, st);
    case 16: return run_stream<CT, QT, D, 16>(p, st);
    case 32: return run_stream<CT, QT, D, 32>(p, st);
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

}  // namespace

// Streaming decode partitions for single-head work items.  Grouped heads go to
// the one-CTA-per-item tensor-core kernel (decode.cu).  (A grouped-head
// variant of this kernel ran a ring of 6 stages for 4 consumer warps, the
// stage-parity race the static_assert on NSTG % NC now rejects, and faulted;
// it is gone.)
cudaError_t launch_decode_stream(const DecodeParams& p, bool mma, cudaStream_t stream)
{
    if (mma)
        return cudaErrorNotSupported;
    if (p.cache_dtype == kF16)
        return stream_simt<kF16, kF16>(p, stream);
    if (p.cache_dtype == kBF16)
        return stream_simt<kBF16, kBF16>(p, stream);
    return p.q_dtype == kF16 ? stream_simt<kE4M3, kF16>(p, stream)
                             : stream_simt<kE4M3, kBF16>(p, stream);
}

}  // namespace pkv
