// prefill.cu -- the prefill entry's shape check and launch choice.
//
// The prompt phase processes all new tokens of a sequence at once
// (「KV Cache从原理到实战」 §2.3); the tensor-core kernel in prefill_ws.cu
// computes it for every supported shape.
#include <cuda_runtime.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

bool prefill_shape_supported(int dtype, int head_dim, int block_size, int group)
{
    return (dtype == kF16 || dtype == kBF16) && (head_dim == 64 || head_dim == 128) &&
           (block_size == 8 || block_size == 16 || block_size == 32) && group >= 1 &&
           group <= 128;
}

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream)
{
    if (!prefill_shape_supported(p.dtype, p.head_dim, p.block_size, p.group))
        return cudaErrorNotSupported;
    if (p.num_seqs <= 0 || p.max_q_len <= 0)
        return cudaSuccess;
    return launch_prefill_ws(p, stream);
}

}  // namespace pkv
