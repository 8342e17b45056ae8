// kv_append.cu -- write each new token's K and V at its slot.
//
// A decode round computes K and V for the new token only and keeps them; the
// token's slot comes from its sequence's block table
// (「KV 缓存与分页注意力」 §02 and §07).  Each thread moves one 16-byte vector
// of the cache: a straight copy when the cache holds the input type, or 16
// inputs scaled by the fp32 reciprocal scale and converted to E4M3 (round to
// nearest even, saturating) for an FP8 cache.  Grid-stride over
// (token, KV head, vector); slots are range-checked before any store.
#include <cuda_runtime.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kAppendThreads = 256;

template <int CT, int IT>
__global__ void __launch_bounds__(kAppendThreads) kv_append_kernel(const AppendParams p)
{
    constexpr int C = Elem<CT>::bytes;
    constexpr int EPV = 16 / C;                      // cache elements per vector
    const int rv = p.head_dim / EPV;                 // vectors per (token, head) row
    const int64_t per_token = (int64_t)p.num_kv_heads * rv;
    const int64_t total = p.num_tokens * per_token;
    const int64_t pool_slots = p.num_blocks * p.block_size;
    // a decode launched after this one may start its set-up now; it waits
    // for this kernel's completion before it reads anything
    pdl_launch_dependents();

    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / per_token;
        const int64_t rem = i - t * per_token;
        const int h = (int)(rem / rv);
        const int cv = (int)(rem - (int64_t)h * rv);
        const int64_t slot = __ldg(p.slot_mapping + t);
        if (slot < 0)
            continue;
        if (slot >= pool_slots) {
            if (h == 0 && cv == 0)
                flag_error(p.dev_err, PKV_DEVERR_SLOT);
            continue;
        }
        const int64_t blk = slot / p.block_size;
        const int64_t off = slot - blk * p.block_size;
        const int64_t dst_elem =
            ((blk * p.num_kv_heads + h) * p.block_size + off) * p.head_dim + (int64_t)cv * EPV;
        const int64_t src_elem = (t * p.num_kv_heads + h) * p.head_dim + (int64_t)cv * EPV;
        const char* ks = reinterpret_cast<const char*>(p.k) + src_elem * 2;
        const char* vs = reinterpret_cast<const char*>(p.v) + src_elem * 2;
        char* kd = reinterpret_cast<char*>(p.k_cache) + dst_elem * C;
        char* vd = reinterpret_cast<char*>(p.v_cache) + dst_elem * C;
        if constexpr (CT == IT) {
            st_v4(kd, ld_ro(ks));
            st_v4(vd, ld_ro(vs));
        } else {
            // 16 inputs -> 16 E4M3 codes
            float kf[16], vf[16];
            unpack_vec<IT>(ld_ro(ks), kf);
            unpack_vec<IT>(ld_ro(ks + 16), kf + 8);
            unpack_vec<IT>(ld_ro(vs), vf);
            unpack_vec<IT>(ld_ro(vs + 16), vf + 8);
            uint32_t kw[4], vw[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint16_t k0 = e4m3x2_satfinite(kf[4 * j] * p.k_inv_scale,
                                                     kf[4 * j + 1] * p.k_inv_scale);
                const uint16_t k1 = e4m3x2_satfinite(kf[4 * j + 2] * p.k_inv_scale,
                                                     kf[4 * j + 3] * p.k_inv_scale);
                const uint16_t v0 = e4m3x2_satfinite(vf[4 * j] * p.v_inv_scale,
                                                     vf[4 * j + 1] * p.v_inv_scale);
                const uint16_t v1 = e4m3x2_satfinite(vf[4 * j + 2] * p.v_inv_scale,
                                                     vf[4 * j + 3] * p.v_inv_scale);
                kw[j] = pack2(k0, k1);
                vw[j] = pack2(v0, v1);
            }
            st_v4(kd, make_uint4(kw[0], kw[1], kw[2], kw[3]));
            st_v4(vd, make_uint4(vw[0], vw[1], vw[2], vw[3]));
        }
    }
}

template <int CT, int IT>
cudaError_t run(const AppendParams& p, cudaStream_t stream)
{
    constexpr int EPV = 16 / Elem<CT>::bytes;
    const int64_t total = p.num_tokens * p.num_kv_heads * (p.head_dim / EPV);
    int64_t blocks = (total + kAppendThreads - 1) / kAppendThreads;
    const int64_t cap = 152 * 16;                    // grid-stride beyond ~16 CTAs per SM
    if (blocks > cap)
        blocks = cap;
    if (blocks <= 0)
        return cudaSuccess;
    kv_append_kernel<CT, IT><<<(unsigned)blocks, kAppendThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream)
{
    if (p.cache_dtype == kF16 && p.in_dtype == kF16)
        return run<kF16, kF16>(p, stream);
    if (p.cache_dtype == kBF16 && p.in_dtype == kBF16)
        return run<kBF16, kBF16>(p, stream);
    if (p.cache_dtype == kE4M3 && p.in_dtype == kF16)
        return run<kE4M3, kF16>(p, stream);
    if (p.cache_dtype == kE4M3 && p.in_dtype == kBF16)
        return run<kE4M3, kBF16>(p, stream);
    return cudaErrorNotSupported;
}

}  // namespace pkv
