// decode_group.cu -- single-pass decode for batches whose sequences share
// leading blocks (forked samples of one prompt, 「KV 缓存与分页注意力」 §08
// 共用，写时复制).
//
// One CTA serves one (group, KV head, row tile): its rows are the group's
// members x the query heads of the KV head, 8 or 16 of them.  A producer warp
// streams, through a ring of shared-memory stages filled by TMA tensor copies,
// first the group's shared blocks (read once, through the first member's
// table, for every row of the tile) and then each member's own blocks after
// the prefix (for that member's rows only).  Three consumer warps take the
// stages in turn and compute, per 16-token sub-block, S^T = K Q^T and
// O^T += V^T P^T with mma.sync (the formulation of the grouped-head kernel in
// decode.cu), keeping an online softmax (fp32, base 2) per row; rows that a
// stage does not belong to get no weight from it.  Each row therefore sees
// exactly the tokens of its own context, prefix first, and the CTA merges its
// warps and writes the output: no partials and no reduce launch.
//
// The stages are 128-byte swizzled (16-byte chunk c of row r of a 64-element
// panel sits at chunk c ^ (r mod 8)), which makes the fragment reads of both
// products free of bank conflicts.  Every mbarrier wait is bounded; after a
// time-out the CTA flags PKV_DEVERR_TIMEOUT, lets its copies land and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "decode_common.cuh"
#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "tc_common.cuh"

namespace pkv {
namespace {

using dec::ceil_div_i;
using dec::kNegInf;

// Three consumer warps, each with two ring stages of a 48 KiB ring (at
// 16 x 128 16-bit tiles): one stage is computed on while the other's copy is
// in flight, and four CTAs still fit on an SM.
constexpr int kNC = 3;                  // consumer warps
constexpr uint32_t kGroupSpin = 1u << 22;
constexpr int kMaxDevices = 64;

// Stage geometry: one (block, KV head) tile of K and one of V, each as D/64
// panels of BS rows x 128 bytes.
template <int D, int BS>
struct GroupShape {
    static constexpr int PANELS = D / 64;
    static constexpr int PANEL = BS * 128;
    static constexpr int TILE = PANELS * PANEL;
    static constexpr int STAGE = 2 * TILE;
    static constexpr int NSTG_RAW = 49152 / STAGE;
    static constexpr int NSTG = NSTG_RAW < kNC ? kNC : (NSTG_RAW > 12 ? 12 : NSTG_RAW / kNC * kNC);
    static constexpr int RING = NSTG * STAGE;
};

// Shared-memory layout, in bytes from the 1024-aligned base.  The warps' merge
// area reuses the ring once every stage has been consumed.
template <int D, int BS, int NNT>
struct GroupSmem {
    using S = GroupShape<D, BS>;
    static constexpr int ROWS = 16;
    static constexpr int MERGE = kNC * ROWS * D * 4 + 2 * kNC * ROWS * 4;
    static constexpr int region = ((S::RING > MERGE ? S::RING : MERGE) + 1023) / 1024 * 1024;
    static constexpr int merge_acc = 0;                              // [kNC][16][D] fp32
    static constexpr int merge_m = kNC * ROWS * D * 4;               // [kNC][16]
    static constexpr int merge_l = merge_m + kNC * ROWS * 4;         // [kNC][16]
    static constexpr int sq = region;                                // Q fragments
    static constexpr int full = sq + NNT * (D / 32) * 32 * 16;
    static constexpr int empty = full + 8 * S::NSTG;
    static constexpr int meta = empty + 8 * S::NSTG;                 // int4 per stage
    static constexpr int misc = meta + 16 * S::NSTG;                 // abort flag, tiles armed
    static constexpr int bytes = misc + 16;
    static constexpr int alloc = bytes + 1024;                       // room to align the base
};

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

__device__ __forceinline__ uint4 lds16(uint32_t addr)
{
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(addr));
    return r;
}

// The 16-byte chunk of a K row (and of q) that lane t of a quad holds for
// k-slice i of the score product: chunks 2t + (i & 1) of 64-dim panel i / 2,
// the same for Q and K (so every dot product is unchanged).  With the
// stage's 128-byte swizzle the eight lanes of a quarter-warp (rows g, g + 1,
// four quads) then read eight distinct 16-byte bank groups.
__device__ __forceinline__ int kchunk(int i, int t)
{
    return 8 * (i >> 1) + 2 * t + (i & 1);
}

__device__ __forceinline__ void consumers_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kNC * 32) : "memory");
}

// Bounded wait for phase `parity` of the mbarrier at `bar`: false when the CTA
// gives up (a time-out here, or one elsewhere in the CTA).  Under a limit
// lowered for testing a poll is one non-suspending look (test_wait), so that a
// one-poll wait that is not already complete always runs out.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, int32_t* dev_err,
                                              uint32_t tries)
{
    const bool look = tries < tc::kSpin;
    WaitClock clock;
    for (uint32_t i = 0; i < tries; ++i) {
        if (look ? tc::test_wait(bar, parity) : tc::try_wait(bar, parity))
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

// The CTA's work, the same for the producer and the consumers.
struct GroupItem {
    int g;            // KV head
    int b0;           // first sequence of the group
    int nmem;         // members this kernel covers
    int row0;         // first row (member x head) of the tile
    int nrows;
    int prefix;       // shared tokens (whole blocks)
    int m_lo, m_hi;   // members with rows in the tile
};

// Segment k of the stream (nseg = 1 + members of the tile): k < nseg - 1
// member m_lo + k after the prefix (its own rows), k = nseg - 1 the shared
// prefix (rows [0, nrows)).  The members' own blocks come first: in a step
// they are the blocks written last (the new tokens), the likeliest to be
// still in L2.  Blocks [blk0, blk1) of `table`, tokens up to t_end; ok =
// false for a member whose context cannot be used (its rows are zeroed at
// the end).
struct Segment {
    const int32_t* table;
    int blk0, blk1;
    int t_end;
    int rlo, rhi;
    bool ok;
};

__device__ __forceinline__ bool member_ok(const DecodeParams& p, int ctx, int prefix)
{
    return ctx >= prefix && ctx <= p.max_context_len &&
           ctx <= p.max_blocks_per_seq * p.block_size;
}

template <int BS>
__device__ __forceinline__ Segment segment(const DecodeParams& p, const GroupItem& it, int k,
                                           int nseg)
{
    Segment sg{};
    const int G = p.group;
    if (k == nseg - 1) {
        sg.table = p.block_tables + (int64_t)it.b0 * p.max_blocks_per_seq;
        sg.blk0 = 0;
        sg.blk1 = it.prefix / BS;
        sg.t_end = it.prefix;
        sg.rlo = 0;
        sg.rhi = it.nrows;
        sg.ok = true;
        return sg;
    }
    const int m = it.m_lo + k;
    const int s = it.b0 + m;
    const int ctx = __ldg(p.context_lens + s);
    sg.ok = member_ok(p, ctx, it.prefix);
    sg.table = p.block_tables + (int64_t)s * p.max_blocks_per_seq;
    sg.blk0 = it.prefix / BS;
    sg.blk1 = sg.ok ? ceil_div_i(ctx, BS) : sg.blk0;
    sg.t_end = ctx;
    sg.rlo = max(m * G - it.row0, 0);
    sg.rhi = min((m + 1) * G - it.row0, it.nrows);
    return sg;
}

// Resident CTAs per SM asked of the compiler: four (a parallel-sampling
// batch's CTAs then fit one wave).
template <int CT, int D, int BS, int NNT>
__global__ void __launch_bounds__((kNC + 1) * 32, 4)
    decode_group_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv)
{
    using S = GroupShape<D, BS>;
    using L = GroupSmem<D, BS, NNT>;
    constexpr bool kBf16 = (CT == kBF16);
    constexpr int NSTG = S::NSTG;
    constexpr int NS = D / 32;          // 32-wide slices of head_dim
    constexpr int NH = D / 64;          // 64-wide panels
    constexpr int NM = D / 16;          // m-tiles of the transposed output
    constexpr int SBB = BS / 16;        // 16-token sub-blocks per block
    constexpr int ROWS = L::ROWS;
    constexpr int RT = 8 * NNT;
    // tile t goes to consumer warp t % kNC and to stage t % NSTG: with NSTG a
    // multiple of kNC the two uses t, t + NSTG of a stage belong to one warp,
    // which waits for t + NSTG only after it has consumed t
    static_assert(NSTG % kNC == 0, "ring stages must be a multiple of the consumer warps");
    static_assert(BS % 16 == 0 && D % 64 == 0, "16-token sub-blocks, 64-dim panels");

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = tc::s_addr(smem_raw);
    unsigned char* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = tc::s_addr(base);
    float* sm_acc = reinterpret_cast<float*>(base + L::merge_acc);
    float* sm_m = reinterpret_cast<float*>(base + L::merge_m);
    float* sm_l = reinterpret_cast<float*>(base + L::merge_l);
    uint4* sq = reinterpret_cast<uint4*>(base + L::sq);
    int4* meta = reinterpret_cast<int4*>(base + L::meta);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L::misc);
    volatile int* armed_rec = reinterpret_cast<volatile int*>(base + L::misc + 4);
    const uint32_t full0 = sbase + L::full;
    const uint32_t empty0 = sbase + L::empty;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int gq = lane >> 2;
    const int t4 = lane & 3;
    const int G = p.group;
    const uint32_t tries = p.wait_tries ? p.wait_tries : kGroupSpin;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTG; ++i) {
            tc::bar_init(full0 + 8 * i, 1);
            tc::bar_init(empty0 + 8 * i, 1);
        }
        *abort_flag = 0;
        *armed_rec = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // launched with programmatic dependent launch: read nothing before the
    // preceding kernel in the stream is complete
    pdl_wait_primary();

    // ------------------------------------------------------------ the item
    GroupItem it{};
    int64_t idx = blockIdx.x;
    it.g = (int)(idx % p.num_kv_heads);
    idx /= p.num_kv_heads;
    const int ntiles = ceil_div_i(p.max_group_size * G, RT);
    const int tile = (int)(idx % ntiles);
    const int grp = (int)(idx / ntiles);
    it.b0 = __ldg(p.grp_begin + grp);
    const int b1 = __ldg(p.grp_begin + grp + 1);
    const int blocks = __ldg(p.grp_prefix_blocks + grp);
    const bool bounds_ok = it.b0 >= 0 && b1 >= it.b0 && b1 <= p.num_seqs;
    if (!bounds_ok || blocks < 0 || blocks > min(p.max_prefix_blocks, p.max_blocks_per_seq)) {
        // an unusable group entry: flagged; with usable bounds its members'
        // rows are zeroed (and flagged as contexts that cannot be used)
        if (it.g == 0 && tile == 0 && threadIdx.x == 0)
            flag_error(p.dev_err, PKV_DEVERR_PREFIX);
        if (bounds_ok && tile == 0) {
            for (int i = threadIdx.x; i < (b1 - it.b0) * G * D; i += blockDim.x) {
                if (i == 0)
                    flag_error(p.dev_err, PKV_DEVERR_CONTEXT);
                dec::store_out<CT>(p, it.b0 + i / (G * D), it.g * G + (i / D) % G, i % D, 0.f);
            }
        }
        return;
    }
    pdl_launch_dependents();
    it.nmem = min(b1 - it.b0, p.max_group_size);
    it.prefix = blocks * BS;
    it.row0 = tile * RT;
    it.nrows = min(RT, it.nmem * G - it.row0);
    // the producer warp starts streaming as soon as the item is known; the
    // consumers do the checks and load q meanwhile
    if (tile == 0 && warp < kNC) {
        // members past max_group_size have no tile: zero their rows
        for (int i = threadIdx.x; i < (b1 - it.b0 - it.nmem) * G * D; i += kNC * 32) {
            const int m = it.nmem + i / (G * D);
            const int h = it.g * G + (i / D) % G;
            if (i % (G * D) == 0)
                flag_error(p.dev_err, PKV_DEVERR_CONTEXT);
            dec::store_out<CT>(p, it.b0 + m, h, i % D, 0.f);
        }
        // every member's table must hold the first member's prefix blocks
        if (it.g == 0) {
            const int32_t* lead = p.block_tables + (int64_t)it.b0 * p.max_blocks_per_seq;
            for (int i = threadIdx.x; i < (it.nmem - 1) * blocks; i += kNC * 32) {
                const int m = 1 + i / blocks;
                const int b = i % blocks;
                if (__ldg(lead + (int64_t)m * p.max_blocks_per_seq + b) != __ldg(lead + b))
                    flag_error(p.dev_err, PKV_DEVERR_PREFIX);
            }
        }
    }
    if (it.nrows <= 0)
        return;
    it.m_lo = it.row0 / G;
    it.m_hi = min(it.nmem, ceil_div_i(it.row0 + it.nrows, G));
    const int nseg = 1 + it.m_hi - it.m_lo;

    // row r of the tile -> (sequence, query head)
    auto row_of = [&](int r) -> int2 {
        const int rho = it.row0 + r;
        return make_int2(it.b0 + rho / G, it.g * G + rho % G);
    };

    // Q^T fragments (rows gq, gq + 8 of the n-tiles; zero past nrows), each
    // lane reading back its own 16 bytes; lane t of a quad holds chunk
    // kchunk(i, t) of k-slice i, as for K (consumer threads only)
    for (int i = threadIdx.x; warp < kNC && i < NNT * NS * 32; i += kNC * 32) {
        const int ln = i & 31;
        const int r = (ln >> 2) + 8 * (i / (NS * 32));
        const int sl = (i >> 5) % NS;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < it.nrows) {
            const int2 sh = row_of(r);
            v = ld_ro(reinterpret_cast<const char*>(p.q) +
                      (((int64_t)sh.x * p.num_heads + sh.y) * D + 8 * kchunk(sl, ln & 3)) * 2);
        }
        sq[i] = v;
    }

    if (warp == kNC) {
        // ------------------------------------------------------------ producer
        uint32_t tt = 0;
        bool stop = false;
        // K/V tiles are read once per call: first out of L2
        const uint64_t kv_policy = l2_evict_first_policy();
        // the first 32 table entries of a segment, one per lane, read before
        // (and without waiting for) the member's context length -- entries
        // past the context are read but not used -- and one segment ahead, so
        // that these round trips overlap the copies before them
        auto first_chunk = [&](const Segment& sg) -> int {
            const int n = min(32, p.max_blocks_per_seq - sg.blk0);
            return lane < n ? __ldg(sg.table + sg.blk0 + lane) : -1;
        };
        Segment sg = segment<BS>(p, it, 0, nseg);
        int next_entry = first_chunk(sg);
        for (int k = 0; k < nseg && !stop; ++k) {
            const int entry0 = next_entry;
            Segment nsg{};
            if (k + 1 < nseg) {
                nsg = segment<BS>(p, it, k + 1, nseg);
                next_entry = first_chunk(nsg);
            }
            for (int c0 = sg.blk0; c0 < sg.blk1 && !stop; c0 += 32) {
                const int n = min(32, sg.blk1 - c0);
                const int entry = c0 == sg.blk0 ? entry0
                                                : (lane < n ? __ldg(sg.table + c0 + lane) : -1);
                for (int j = 0; j < n; ++j) {
                    const int phys = __shfl_sync(0xffffffffu, entry, j);
                    const uint32_t stage = tt % NSTG;
                    const uint32_t use = tt / NSTG;
                    const bool valid = phys >= 0 && (int64_t)phys < p.num_blocks;
                    int ok = 1;
                    if (lane == 0) {
                        ok = use == 0 || wait_or_abort(empty0 + 8 * stage, (use - 1) & 1,
                                                       abort_flag, p.dev_err, tries);
                        if (ok) {
                            meta[stage] = make_int4(sg.rlo | (sg.rhi << 8) | ((int)valid << 16),
                                                    (c0 + j) * BS, sg.t_end, 0);
                            const uint32_t fb = full0 + 8 * stage;
                            if (valid) {
                                asm volatile(
                                    "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                                        fb),
                                    "r"((uint32_t)S::STAGE)
                                    : "memory");
                                const uint32_t dst = sbase + stage * S::STAGE;
                                const int y = (int)(((int64_t)phys * p.num_kv_heads + it.g) * BS);
#pragma unroll
                                for (int pn = 0; pn < S::PANELS; ++pn) {
                                    tc::tma_box_hint(dst + pn * S::PANEL, &tmk, pn * 64, y, fb,
                                                     kv_policy);
                                    tc::tma_box_hint(dst + S::TILE + pn * S::PANEL, &tmv, pn * 64,
                                                     y, fb, kv_policy);
                                }
                            } else {
                                flag_error(p.dev_err, PKV_DEVERR_BLOCK_ID);
                                tc::bar_arrive(fb);
                            }
                            *armed_rec = (int)(tt + 1);
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    ++tt;
                    if (!ok) {
                        stop = true;
                        break;
                    }
                }
            }
            sg = nsg;
        }
    } else {
        // ------------------------------------------------------------ consumers
        consumers_sync();                       // q fragments are in shared memory
        // tiles of the whole stream, counted the producer's way
        uint32_t ntile = 0;
        for (int k = 0; k < nseg; ++k) {
            const Segment sg = segment<BS>(p, it, k, nseg);
            ntile += (uint32_t)(sg.blk1 - sg.blk0);
        }
        const float qk = p.qk_scale_log2;
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

        for (uint32_t tt = warp; tt < ntile; tt += kNC) {
            const uint32_t stage = tt % NSTG;
            const bool ok = __all_sync(0xffffffffu,
                                       wait_or_abort(full0 + 8 * stage, (tt / NSTG) & 1,
                                                     abort_flag, p.dev_err, tries));
            const int4 md = meta[stage];
            if (ok && ((md.x >> 16) & 1)) {
                const int rlo = md.x & 0xff;
                const int rhi = (md.x >> 8) & 0xff;
                const int t_end = md.z;
                const uint32_t ks = sbase + stage * S::STAGE;
                const uint32_t vs = ks + S::TILE;
                // rows of this lane's accumulators: 8n + 2 t4 + h
                bool row_in[NNT][2];
#pragma unroll
                for (int n = 0; n < NNT; ++n)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int r = 8 * n + 2 * t4 + h;
                        row_in[n][h] = r >= rlo && r < rhi;
                    }
#pragma unroll 1
                for (int sb = 0; sb < SBB; ++sb) {
                    const int tb = md.y + sb * 16;       // first token of the sub-block
                    if (tb >= t_end)
                        break;
                    // S^T = K Q^T: rows = tokens tb + gq (+ 8)
                    float sc[NNT][4];
#pragma unroll
                    for (int n = 0; n < NNT; ++n)
                        sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
                    const int kr0 = sb * 16 + gq;
#pragma unroll
                    for (int i2 = 0; i2 < NS; ++i2) {
                        const int c = kchunk(i2, t4);              // 16-byte chunk of the row
                        const uint4 k0 = lds16(ks + tc::panel_off(kr0, c, BS));
                        const uint4 k1 = lds16(ks + tc::panel_off(kr0 + 8, c, BS));
                        uint4 qv[NNT];
#pragma unroll
                        for (int n = 0; n < NNT; ++n)
                            qv[n] = ld_shared16(sq + (n * NS + i2) * 32 + lane);
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const uint32_t a[4] = {reg_of(k0, 2 * u), reg_of(k1, 2 * u),
                                                   reg_of(k0, 2 * u + 1), reg_of(k1, 2 * u + 1)};
#pragma unroll
                            for (int n = 0; n < NNT; ++n)
                                mma16816(sc[n], a, reg_of(qv[n], 2 * u),
                                         reg_of(qv[n], 2 * u + 1), kBf16);
                        }
                    }
                    // online softmax (base 2); sc[n][e] is token tb + gq + 8 (e >> 1),
                    // row 8n + 2 t4 + (e & 1)
                    float x[NNT][4];
                    float mn[NNT][2];
                    bool raise = false;
#pragma unroll
                    for (int n = 0; n < NNT; ++n) {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            x[n][e] = (row_in[n][e & 1] && tb + gq + 8 * (e >> 1) < t_end)
                                          ? sc[n][e] * qk
                                          : kNegInf;
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
                                // a row that has seen no token yet keeps its zeros
                                al[n][h] = mn[n][h] == kNegInf ? 1.f : exp2f(m_h[n][h] - mn[n][h]);
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
                    // P^T fragments through 8x8 transposes (see decode.cu)
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
                                bl[n][hf] = transpose8x8(
                                    pack2(round_to<kBF16>(r0), round_to<kBF16>(r1)));
                            } else {
                                bh[n][hf] =
                                    transpose8x8(pack2(round_to<kF16>(v0), round_to<kF16>(v1)));
                                bl[n][hf] = 0u;
                            }
                        }
                    // O^T += V^T P^T, one 64-dim panel at a time: V rows of tokens
                    // 2 t4, 2 t4 + 1, 2 t4 + 8, 2 t4 + 9, dims 64 hv + 8 gq + [0, 8)
#pragma unroll
                    for (int hv = 0; hv < NH; ++hv) {
                        uint4 vc[4];
#pragma unroll
                        for (int tk = 0; tk < 4; ++tk) {
                            const int vr = 2 * t4 + (tk & 1) + 8 * (tk >> 1);
                            vc[tk] = lds16(vs + tc::panel_off(sb * 16 + vr, 8 * hv + gq, BS));
                            // tokens past the range get p = 0; clear their V so that
                            // whatever bits sit in those slots cannot make NaN
                            if (tb + vr >= t_end)
                                vc[tk] = make_uint4(0, 0, 0, 0);
                        }
#pragma unroll
                        for (int e4 = 0; e4 < 4; ++e4) {
                            const int j = 4 * hv + e4;
                            const uint32_t lo0 = reg_of(vc[0], e4), lo1 = reg_of(vc[1], e4);
                            const uint32_t hi0 = reg_of(vc[2], e4), hi1 = reg_of(vc[3], e4);
                            const uint32_t a[4] = {__byte_perm(lo0, lo1, 0x5410),
                                                   __byte_perm(lo0, lo1, 0x7632),
                                                   __byte_perm(hi0, hi1, 0x5410),
                                                   __byte_perm(hi0, hi1, 0x7632)};
#pragma unroll
                            for (int n = 0; n < NNT; ++n) {
                                mma16816(acc[j][n], a, bh[n][0], bh[n][1], kBf16);
                                if constexpr (kBf16)
                                    mma16816(acc[j][n], a, bl[n][0], bl[n][1], kBf16);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (ok && lane == 0)
                tc::bar_arrive(empty0 + 8 * stage);
        }

        // head sums over the eight lanes of a row
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
        // every consumer warp is done with the ring: it becomes the merge area
        consumers_sync();
        if (gq == 0) {
#pragma unroll
            for (int n = 0; n < NNT; ++n)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    sm_m[warp * ROWS + 8 * n + 2 * t4 + h] = m_h[n][h];
                    sm_l[warp * ROWS + 8 * n + 2 * t4 + h] = l_h[n][h];
                }
        }
        // accumulator (j, n, e): row 8n + 2 t4 + (e & 1),
        // dim 64 (j / 4) + 8 gq + 2 (j % 4) + (e >> 1)
#pragma unroll
        for (int j = 0; j < NM; ++j)
#pragma unroll
            for (int n = 0; n < NNT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int row = 8 * n + 2 * t4 + (e & 1);
                    const int d = 64 * (j >> 2) + 8 * gq + 2 * (j & 3) + (e >> 1);
                    sm_acc[(warp * ROWS + row) * D + d] = acc[j][n][e];
                }
        consumers_sync();
        // merge the warps and write every row of the tile; a member whose
        // context cannot be used gets zeros and a flag
        const int tid = threadIdx.x;
        for (int i = tid; i < it.nrows * D; i += kNC * 32) {
            const int row = i / D;
            const int d = i % D;
            const int2 sh = row_of(row);
            const int ctx = __ldg(p.context_lens + sh.x);
            if (!member_ok(p, ctx, it.prefix)) {
                if (d == 0 && sh.y == it.g * G)
                    flag_error(p.dev_err, PKV_DEVERR_CONTEXT);
                dec::store_out<CT>(p, sh.x, sh.y, d, 0.f);
                continue;
            }
            float M = kNegInf;
#pragma unroll
            for (int k = 0; k < kNC; ++k)
                M = fmaxf(M, sm_m[k * ROWS + row]);
            float Lsum = 0.f;
            float O = 0.f;
            if (M != kNegInf) {
#pragma unroll
                for (int k = 0; k < kNC; ++k) {
                    const float mk = sm_m[k * ROWS + row];
                    if (mk != kNegInf) {
                        const float f = exp2f(mk - M);
                        Lsum += sm_l[k * ROWS + row] * f;
                        O += sm_acc[(k * ROWS + row) * D + d] * f;
                    }
                }
            }
            dec::store_out<CT>(p, sh.x, sh.y, d, Lsum > 0.f ? O / Lsum : 0.f);
        }
    }
    // Every copy this CTA started lands before it exits: without a time-out
    // the consumers waited for each one; after one, the last NSTG stages armed
    // may still be in flight (the producer's record is final at this barrier).
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        const uint32_t armed = (uint32_t)*armed_rec;
        const uint32_t first = armed > (uint32_t)NSTG ? armed - NSTG : 0;
        for (uint32_t tt = first; tt < armed; ++tt) {
            WaitClock clock;
            for (uint32_t i = 0; i < kGroupSpin; ++i)
                if (tc::try_wait(full0 + 8 * (tt % NSTG), (tt / NSTG) & 1) || clock.expired(i))
                    break;
        }
    }
}

// ------------------------------------------------------------------ dispatch

template <int CT, int D, int BS, int NNT>
cudaError_t run_group(const DecodeParams& p, cudaStream_t stream)
{
    using L = GroupSmem<D, BS, NNT>;
    auto kern = decode_group_kernel<CT, D, BS, NNT>;
    // the shared-memory opt-in, once per device
    static std::atomic<int> opted[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    if (!opted[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::alloc);
        if (e != cudaSuccess)
            return e;
        opted[dev].store(1, std::memory_order_release);
    }
    const int64_t rows = p.num_blocks * p.num_kv_heads * BS;
    CUtensorMap tmk, tmv;
    if (!tc::cache_map(&tmk, p.k_cache, rows, D, BS) ||
        !tc::cache_map(&tmv, p.v_cache, rows, D, BS))
        return cudaErrorNotSupported;
    const int RT = 8 * NNT;
    const int64_t ntiles = ((int64_t)p.max_group_size * p.group + RT - 1) / RT;
    const int64_t ctas = (int64_t)p.num_groups * ntiles * p.num_kv_heads;
    if (ctas <= 0)
        return cudaSuccess;
    if (ctas > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3((kNC + 1) * 32);
    cfg.dynamicSmemBytes = L::alloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, tmk, tmv);
}

template <int CT, int D, int BS>
cudaError_t group_rows(const DecodeParams& p, cudaStream_t st)
{
    return (int64_t)p.max_group_size * p.group > 8 ? run_group<CT, D, BS, 2>(p, st)
                                                    : run_group<CT, D, BS, 1>(p, st);
}

template <int CT>
cudaError_t group_shape(const DecodeParams& p, cudaStream_t st)
{
    if (p.head_dim == 64 && p.block_size == 16) return group_rows<CT, 64, 16>(p, st);
    if (p.head_dim == 64 && p.block_size == 32) return group_rows<CT, 64, 32>(p, st);
    if (p.head_dim == 128 && p.block_size == 16) return group_rows<CT, 128, 16>(p, st);
    if (p.head_dim == 128 && p.block_size == 32) return group_rows<CT, 128, 32>(p, st);
    return cudaErrorNotSupported;
}

}  // namespace

int64_t group_decode_ctas(const DecodeParams& p)
{
    const int64_t rows = (int64_t)p.max_group_size * p.group;
    const int rt = rows > 8 ? 16 : 8;
    return (int64_t)p.num_groups * ((rows + rt - 1) / rt) * p.num_kv_heads;
}

cudaError_t launch_decode_group(const DecodeParams& p, cudaStream_t stream)
{
    if (!prefix_kernel_supported(p.cache_dtype, p.q_dtype, p.head_dim, p.block_size, p.group))
        return cudaErrorNotSupported;
    if (p.grp_begin == nullptr || p.num_groups <= 0 || p.max_group_size <= 0)
        return cudaErrorInvalidValue;
    return p.cache_dtype == kF16 ? group_shape<kF16>(p, stream) : group_shape<kBF16>(p, stream);
}

}  // namespace pkv
