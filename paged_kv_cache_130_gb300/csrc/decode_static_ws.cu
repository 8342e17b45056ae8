// decode_static_ws.cu -- decode attention for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc or hand the library a scratch buffer: an
// engine that has reserved nearly all of the GPU's memory up front for its own
// KV-cache pool (a cudaMalloc would then fail), or code on a latency-critical
// path where cudaMalloc / cudaFree may synchronise the device.  This entry
// point runs the same decode as pkv_paged_attention_decode but takes the
// split-context partials from a static device array inside the library.  It
// allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
#include <cuda_runtime.h>

#include <mutex>

#include "pkv.h"

namespace {

constexpr size_t kScratchBytes = PKV_STATIC_SCRATCH_BYTES;

// The scratch itself.  Every GPU that loads the library holds it until the
// process exits.  On the host, this name is only a stand-in for the symbol,
// never a device address: the address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
pkv_status scratch_address(void** addr)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess || p == nullptr)
            return PKV_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_paged_attention_decode_static_ws(
    const pkv_cache_desc* cache, const void* q, int32_t q_dtype, int32_t num_seqs,
    int32_t num_heads, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* context_lens, int32_t max_context_len, float scale, int32_t partition_size,
    int32_t* dev_err, void* out, pkv_stream_t stream)
{
    // the partials this request needs; larger than the static array -> refuse
    const size_t need = pkv_decode_workspace_bytes(cache, num_seqs, num_heads, max_context_len,
                                                   partition_size);
    if (need > kScratchBytes)
        return PKV_ERR_SCRATCH_LIMIT;
    void* ws = nullptr;
    if (need > 0) {
        const pkv_status st = scratch_address(&ws);
        if (st != PKV_OK)
            return st;
    }
    // Nothing in the scratch has to start at zero: the partition kernel writes
    // every partial (m, l, o) that the reduce kernel of the same call reads.
    return pkv_paged_attention_decode(cache, q, q_dtype, num_seqs, num_heads, block_tables,
                                      max_blocks_per_seq, context_lens, max_context_len, scale,
                                      partition_size, ws, need > 0 ? kScratchBytes : 0, dev_err,
                                      out, stream);
}
