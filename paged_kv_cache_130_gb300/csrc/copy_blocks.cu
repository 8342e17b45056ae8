// copy_blocks.cu -- copy-on-write block copy.
//
// Before a sequence writes into a block it shares with others, the block is
// copied and the write goes to the copy (「KV 缓存与分页注意力」 §08).  A block
// is num_kv_heads * block_size * head_dim elements of K and as many of V, one
// contiguous run each.  Grid: x = 16-KiB chunk of a block, y = (layer, K|V),
// z = pair; each thread moves 4 vectors of 16 bytes, all loads before the
// stores.  Pair ids are range-checked before any access.
#include <cuda_runtime.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kVecPerThread = 4;
constexpr int64_t kChunkBytes = (int64_t)kCopyThreads * kVecPerThread * 16;   // 16 KiB

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(const CopyParams p)
{
    const int64_t pair = blockIdx.z;
    const int layer = blockIdx.y >> 1;
    const bool is_v = blockIdx.y & 1;
    const int64_t src = __ldg(p.pairs + 2 * pair);
    const int64_t dst = __ldg(p.pairs + 2 * pair + 1);
    if (src < 0 || src >= p.num_blocks || dst < 0 || dst >= p.num_blocks) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
            flag_error(p.dev_err, PKV_DEVERR_COPY_PAIR);
        return;
    }
    char* base = reinterpret_cast<char*>(is_v ? p.v[layer] : p.k[layer]);
    const char* s = base + src * p.block_bytes;
    char* d = base + dst * p.block_bytes;
    const int64_t start = (int64_t)blockIdx.x * kChunkBytes;
    uint4 buf[kVecPerThread];
#pragma unroll
    for (int j = 0; j < kVecPerThread; ++j) {
        const int64_t off = start + ((int64_t)j * kCopyThreads + threadIdx.x) * 16;
        if (off < p.block_bytes)
            buf[j] = ld_stream(s + off);
    }
#pragma unroll
    for (int j = 0; j < kVecPerThread; ++j) {
        const int64_t off = start + ((int64_t)j * kCopyThreads + threadIdx.x) * 16;
        if (off < p.block_bytes)
            st_v4(d + off, buf[j]);
    }
}

}  // namespace

cudaError_t launch_copy_blocks(const CopyParams& p, cudaStream_t stream)
{
    if (p.num_pairs <= 0 || p.num_layers <= 0)
        return cudaSuccess;
    if (p.num_pairs > 65535 || p.num_layers > kCopyMaxLayers)
        return cudaErrorInvalidConfiguration;
    const int64_t chunks = (p.block_bytes + kChunkBytes - 1) / kChunkBytes;
    if (chunks > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)chunks, (unsigned)(2 * p.num_layers), (unsigned)p.num_pairs);
    copy_blocks_kernel<<<grid, kCopyThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv
