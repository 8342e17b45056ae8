// swap.cu -- block swap between the device cache and host memory.
//
// When the pool runs short, all blocks of a pre-empted sequence move to CPU
// memory and come back when it is scheduled again (「KV 缓存与分页注意力」 §09).
// GB300 reaches pinned Grace memory over NVLink-C2C with ordinary loads and
// stores, so one kernel moves every (src block, dst block) pair of every layer
// in one launch, whichever side is the host: no per-block copy calls.  Grid:
// x = 16-KiB chunk of a block, y = (layer, K|V), z = pair; each thread issues
// its four 16-byte loads before its stores.  Pair ids are range-checked
// against their own pool before any access.
#include <cuda_runtime.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kSwapThreads = 256;
constexpr int kSwapVec = 4;
constexpr int64_t kSwapChunk = (int64_t)kSwapThreads * kSwapVec * 16;   // 16 KiB

__global__ void __launch_bounds__(kSwapThreads) swap_blocks_kernel(const SwapParams p)
{
    const int64_t pair = blockIdx.z;
    const int layer = blockIdx.y >> 1;
    const bool is_v = blockIdx.y & 1;
    const int64_t src = __ldg(p.pairs + 2 * pair);
    const int64_t dst = __ldg(p.pairs + 2 * pair + 1);
    if (src < 0 || src >= p.src_blocks || dst < 0 || dst >= p.dst_blocks) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
            flag_error(p.dev_err, PKV_DEVERR_COPY_PAIR);
        return;
    }
    const char* s = reinterpret_cast<const char*>(is_v ? p.src_v[layer] : p.src_k[layer]) +
                    src * p.block_bytes;
    char* d = reinterpret_cast<char*>(is_v ? p.dst_v[layer] : p.dst_k[layer]) +
              dst * p.block_bytes;
    const int64_t start = (int64_t)blockIdx.x * kSwapChunk;
    uint4 buf[kSwapVec];
#pragma unroll
    for (int j = 0; j < kSwapVec; ++j) {
        const int64_t off = start + ((int64_t)j * kSwapThreads + threadIdx.x) * 16;
        if (off < p.block_bytes)
            buf[j] = *reinterpret_cast<const uint4*>(s + off);
    }
#pragma unroll
    for (int j = 0; j < kSwapVec; ++j) {
        const int64_t off = start + ((int64_t)j * kSwapThreads + threadIdx.x) * 16;
        if (off < p.block_bytes)
            st_v4(d + off, buf[j]);
    }
}

// A plain streaming copy with SM loads and stores: every thread moves
// kProbeVec 16-byte vectors per round (all loads before the stores), rounds
// striding over the whole grid.  It measures what SMs reach over a link (for
// instance device memory <-> pinned host memory over NVLink-C2C), the ceiling
// a copy kernel such as swap_blocks_kernel can aim for.
constexpr int kProbeThreads = 256;
constexpr int kProbeVec = 8;

__global__ void __launch_bounds__(kProbeThreads) stream_copy_kernel(uint4* dst, const uint4* src,
                                                                    int64_t n16)
{
    const int64_t stride = (int64_t)gridDim.x * kProbeThreads * kProbeVec;
    for (int64_t base = (int64_t)blockIdx.x * kProbeThreads * kProbeVec; base < n16;
         base += stride) {
        uint4 buf[kProbeVec];
#pragma unroll
        for (int j = 0; j < kProbeVec; ++j) {
            const int64_t i = base + (int64_t)j * kProbeThreads + threadIdx.x;
            if (i < n16)
                buf[j] = src[i];
        }
#pragma unroll
        for (int j = 0; j < kProbeVec; ++j) {
            const int64_t i = base + (int64_t)j * kProbeThreads + threadIdx.x;
            if (i < n16)
                dst[i] = buf[j];
        }
    }
}

}  // namespace

cudaError_t launch_stream_copy(void* dst, const void* src, int64_t bytes, cudaStream_t stream)
{
    if (bytes <= 0)
        return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    const int64_t n16 = bytes / 16;
    const int64_t per_cta = (int64_t)kProbeThreads * kProbeVec;
    int64_t ctas = (n16 + per_cta - 1) / per_cta;
    if (ctas > 4LL * sms)
        ctas = 4LL * sms;
    stream_copy_kernel<<<(unsigned)ctas, kProbeThreads, 0, stream>>>(
        reinterpret_cast<uint4*>(dst), reinterpret_cast<const uint4*>(src), n16);
    return cudaGetLastError();
}

cudaError_t launch_swap_blocks(const SwapParams& p, cudaStream_t stream)
{
    if (p.num_pairs <= 0 || p.num_layers <= 0)
        return cudaSuccess;
    if (p.num_pairs > 65535 || p.num_layers > kCopyMaxLayers)
        return cudaErrorInvalidConfiguration;
    const int64_t chunks = (p.block_bytes + kSwapChunk - 1) / kSwapChunk;
    if (chunks > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)chunks, (unsigned)(2 * p.num_layers), (unsigned)p.num_pairs);
    swap_blocks_kernel<<<grid, kSwapThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv
