// block_hash.cu -- chained content hashes of full blocks (prefix caching).
//
// Prefix caching gives every full block a hash of its tokens and of all the
// content in front of it, so that requests with the same opening find the same
// blocks (「KV 缓存与分页注意力」 §11; 「KV Cache从原理到实战」 §4.2).  Block i of
// a sequence gets
//   h_i = SHA-256(h_{i-1} || token ids of block i, little-endian int32)
// with h_{-1} the sequence's parent hash (zeros when none is given).  The
// chain is sequential inside a sequence, so one thread walks one sequence;
// sequences run in parallel.  SHA-256 is written from FIPS 180-4: the round
// constants and the initial state are derived on the host from their
// definition (fractional bits of cube and square roots of the first primes)
// with exact integer arithmetic and passed as a kernel parameter.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ __forceinline__ uint32_t rotr(uint32_t x, int n) { return __funnelshift_r(x, x, n); }

__device__ __forceinline__ uint32_t bswap32(uint32_t x) { return __byte_perm(x, 0, 0x0123); }

// One SHA-256 compression of the 16-word chunk w into the state st.
__device__ __forceinline__ void sha256_compress(uint32_t (&st)[8], uint32_t (&w)[16],
                                                const Sha256Table& t)
{
    uint32_t a = st[0], b = st[1], c = st[2], d = st[3];
    uint32_t e = st[4], f = st[5], g = st[6], h = st[7];
#pragma unroll
    for (int i = 0; i < 64; ++i) {
        uint32_t wi;
        if (i < 16) {
            wi = w[i];
        } else {
            const uint32_t x15 = w[(i + 1) & 15];      // W[i-15]
            const uint32_t x2 = w[(i + 14) & 15];      // W[i-2]
            const uint32_t s0 = rotr(x15, 7) ^ rotr(x15, 18) ^ (x15 >> 3);
            const uint32_t s1 = rotr(x2, 17) ^ rotr(x2, 19) ^ (x2 >> 10);
            wi = w[i & 15] + s0 + w[(i + 9) & 15] + s1;  // + W[i-16] + W[i-7]
            w[i & 15] = wi;
        }
        const uint32_t t1 = h + (rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25)) + ((e & f) ^ (~e & g)) +
                            t.k[i] + wi;
        const uint32_t t2 = (rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22)) + ((a & b) ^ (a & c) ^ (b & c));
        h = g;
        g = f;
        f = e;
        e = d + t1;
        d = c;
        c = b;
        b = a;
        a = t1 + t2;
    }
    st[0] += a;
    st[1] += b;
    st[2] += c;
    st[3] += d;
    st[4] += e;
    st[5] += f;
    st[6] += g;
    st[7] += h;
}

// Message of one block: 8 parent words, BS token words, the 0x80 marker, zero
// fill and the 64-bit big-endian bit length; NCH 64-byte chunks.
template <int BS>
__global__ void __launch_bounds__(128) block_hash_kernel(const HashParams p)
{
    constexpr int NW = 8 + BS;                         // data words
    constexpr int NCH = (NW * 4 + 9 + 63) / 64;        // chunks after padding
    constexpr uint32_t kBits = NW * 32;
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= p.num_seqs)
        return;
    const int64_t b0 = __ldg(p.cu_seqlens + s);
    const int64_t b1 = __ldg(p.cu_seqlens + s + 1);
    if (b0 < 0 || b1 < b0 || b1 > p.total_tokens) {
        flag_error(p.dev_err, PKV_DEVERR_CONTEXT);
        return;
    }
    const int64_t nfull = (b1 - b0) / BS;
    const int64_t off = __ldg(p.block_offsets + s);
    if (off < 0 || off + nfull > p.total_blocks) {
        flag_error(p.dev_err, PKV_DEVERR_CONTEXT);
        return;
    }
    uint32_t par[8];
    if (p.parent_hashes != nullptr) {
        const uint4* ph = reinterpret_cast<const uint4*>(p.parent_hashes + (int64_t)s * 32);
        const uint4 x = __ldg(ph), y = __ldg(ph + 1);
        const uint32_t raw[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
            par[i] = bswap32(raw[i]);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            par[i] = 0u;
    }
    const int32_t* tok = p.token_ids + b0;
    // the token words of block blk + 1 are read while block blk is hashed, so
    // the chain does not wait for memory between blocks
    uint32_t cur[BS];
#pragma unroll
    for (int i = 0; i < BS; ++i)
        cur[i] = nfull > 0 ? (uint32_t)__ldg(tok + i) : 0u;
    for (int64_t blk = 0; blk < nfull; ++blk) {
        uint32_t nxt[BS];
        const bool more = blk + 1 < nfull;
#pragma unroll
        for (int i = 0; i < BS; ++i)
            nxt[i] = more ? (uint32_t)__ldg(tok + (blk + 1) * BS + i) : 0u;
        uint32_t st[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            st[i] = p.table.h0[i];
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int j = ch * 16 + i;             // word of the padded message
                uint32_t v = 0u;
                if (j < 8)
                    v = par[j];
                else if (j < NW)
                    v = bswap32(cur[j - 8]);
                else if (j == NW)
                    v = 0x80000000u;
                else if (j == NCH * 16 - 1)
                    v = kBits;
                w[i] = v;
            }
            sha256_compress(st, w, p.table);
        }
        uint32_t* dst = reinterpret_cast<uint32_t*>(p.hashes + (off + blk) * 32);
        uint4 lo, hi;
        lo.x = bswap32(st[0]);
        lo.y = bswap32(st[1]);
        lo.z = bswap32(st[2]);
        lo.w = bswap32(st[3]);
        hi.x = bswap32(st[4]);
        hi.y = bswap32(st[5]);
        hi.z = bswap32(st[6]);
        hi.w = bswap32(st[7]);
        reinterpret_cast<uint4*>(dst)[0] = lo;
        reinterpret_cast<uint4*>(dst)[1] = hi;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            par[i] = st[i];
#pragma unroll
        for (int i = 0; i < BS; ++i)
            cur[i] = nxt[i];
    }
}

// floor(2^32 * frac(root)) where root is the n-th root (n = 2 or 3) of the
// prime p: the largest x with x^n <= p * 2^(32 n), less its integer part.
uint32_t root_fraction_bits(uint32_t p, int n)
{
    using u128 = unsigned __int128;
    const u128 target = (u128)p << (32 * n);
    uint64_t lo = 0, hi = (uint64_t)1 << 40;         // 2^40 > p^(1/n) * 2^32 for p < 2^16
    while (hi - lo > 1) {
        const uint64_t mid = lo + (hi - lo) / 2;
        u128 v = 1;
        for (int i = 0; i < n; ++i)
            v *= (u128)mid;
        if (v <= target)
            lo = mid;
        else
            hi = mid;
    }
    return (uint32_t)(lo & 0xffffffffu);
}

}  // namespace

const Sha256Table& sha256_table()
{
    static Sha256Table table;
    static std::once_flag once;
    std::call_once(once, [] {
        uint32_t primes[64];
        int n = 0;
        for (uint32_t c = 2; n < 64; ++c) {
            bool prime = true;
            for (uint32_t d = 2; d * d <= c; ++d)
                if (c % d == 0) {
                    prime = false;
                    break;
                }
            if (prime)
                primes[n++] = c;
        }
        for (int i = 0; i < 64; ++i)
            table.k[i] = root_fraction_bits(primes[i], 3);
        for (int i = 0; i < 8; ++i)
            table.h0[i] = root_fraction_bits(primes[i], 2);
    });
    return table;
}

cudaError_t launch_block_hashes(const HashParams& p, cudaStream_t stream)
{
    if (p.num_seqs <= 0)
        return cudaSuccess;
    const unsigned grid = (unsigned)((p.num_seqs + 127) / 128);
    switch (p.block_size) {
    case 8: block_hash_kernel<8><<<grid, 128, 0, stream>>>(p); break;
    case 16: block_hash_kernel<16><<<grid, 128, 0, stream>>>(p); break;
    case 32: block_hash_kernel<32><<<grid, 128, 0, stream>>>(p); break;
    default: return cudaErrorNotSupported;
    }
    return cudaGetLastError();
}

}  // namespace pkv
