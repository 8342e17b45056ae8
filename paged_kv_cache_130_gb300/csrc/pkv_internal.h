// pkv_internal.h -- launch interface between the C ABI (pkv_api.cu) and the
// kernel translation units.  Not installed; not part of the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

struct DecodeParams {
    const void* k_cache;
    const void* v_cache;
    int64_t num_blocks;
    int32_t num_kv_heads;
    int32_t block_size;
    int32_t head_dim;
    int32_t cache_dtype;
    float k_scale;
    float v_scale;
    const void* q;
    int32_t q_dtype;
    int32_t num_seqs;
    int32_t num_heads;
    int32_t group;                 // num_heads / num_kv_heads
    const int32_t* block_tables;
    int32_t max_blocks_per_seq;
    const int32_t* context_lens;
    int32_t max_context_len;
    int32_t partition_size;
    int32_t max_partitions;        // partials per (sequence, head) row of the workspace
    int32_t grid_partitions;       // ceil(max_context_len / partition_size)
    float qk_scale_log2;           // scale * log2(e) * k_scale
    float* ws_m;
    float* ws_l;
    float* ws_o;
    int32_t* dev_err;
    void* out;
    // Shared prefixes (all null / 0 for a plain decode): sequences
    // [grp_begin[i], grp_begin[i + 1]) share their first grp_prefix_blocks[i]
    // blocks.  The prefix kernel covers the first max_group_size members of a
    // group and prefixes of up to max_prefix_blocks blocks.
    const int32_t* grp_begin;
    const int32_t* grp_prefix_blocks;
    int32_t num_groups;
    int32_t max_group_size;
    int32_t max_prefix_blocks;
    int32_t prefix_partition;      // tokens per partition of a shared prefix
    // Set when the prefix kernel runs just before: the partition kernel is
    // then launched with programmatic dependent launch, overlaps it, and waits
    // for it (griddepcontrol.wait) only before its CTAs exit, so that its own
    // completion implies the prefix kernel's.
    int32_t wait_prior;
    // Polls per bounded mbarrier wait of the streaming kernel's ring and item
    // queue; 0 = the kernel's own limit.  Only tests set it (to make a wait
    // run out on purpose); the drain of copies in flight ignores it.
    uint32_t wait_tries;
};

// Process-wide wait-limit setting that the decode entry points copy into
// DecodeParams::wait_tries (pkv_testing_set_decode_wait_limit).
uint32_t decode_wait_tries();

struct ReduceParams {
    int32_t num_seqs;
    int32_t num_heads;
    int32_t head_dim;
    const int32_t* context_lens;
    int32_t max_context_len;
    int32_t partition_size;
    int32_t max_partitions;
    const float* ws_m;
    const float* ws_l;
    const float* ws_o;
    int32_t out_dtype;
    void* out;
    int32_t block_size;
    const int32_t* grp_begin;            // shared prefixes, as in DecodeParams
    const int32_t* grp_prefix_blocks;
    int32_t num_groups;
    int32_t max_group_size;
    int32_t max_prefix_blocks;
    int32_t prefix_partition;
};

struct AppendParams {
    void* k_cache;
    void* v_cache;
    int64_t num_blocks;
    int32_t num_kv_heads;
    int32_t block_size;
    int32_t head_dim;
    int32_t cache_dtype;
    float k_inv_scale;
    float v_inv_scale;
    const void* k;
    const void* v;
    int32_t in_dtype;
    const int64_t* slot_mapping;
    int64_t num_tokens;
    int32_t* dev_err;
};

constexpr int kCopyMaxLayers = 64;

struct PrefillParams {
    const void* k_cache;
    const void* v_cache;
    int64_t num_blocks;
    int32_t num_kv_heads;
    int32_t block_size;
    int32_t head_dim;
    int32_t dtype;                 // cache, q and out (F16 or BF16)
    const void* q;                 // [total_q][num_heads][head_dim]
    int32_t num_seqs;
    int32_t num_heads;
    int32_t group;
    const int32_t* cu_seqlens_q;   // [num_seqs + 1]
    int32_t total_q;               // rows of q and out
    int32_t max_q_len;
    const int32_t* block_tables;
    int32_t max_blocks_per_seq;
    const int32_t* context_lens;
    int32_t max_context_len;
    float qk_scale_log2;           // scale * log2(e)
    int32_t* dev_err;
    void* out;                     // [total_q][num_heads][head_dim]
};

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream);
cudaError_t launch_prefill_ws(const PrefillParams& p, cudaStream_t stream);
bool prefill_shape_supported(int dtype, int head_dim, int block_size, int group);

// Partitions of a shared prefix: prefix_partition = max(partition_size,
// round_up(ceil(max_prefix_tokens / kPrefixParts), block_size)) tokens, so no
// row has more than kPrefixParts prefix partials.
constexpr int kPrefixParts = 4;

struct CopyParams {
    void* k[kCopyMaxLayers];
    void* v[kCopyMaxLayers];
    int32_t num_layers;
    int64_t num_blocks;
    int64_t block_bytes;
    const int64_t* pairs;
    int64_t num_pairs;
    int32_t* dev_err;
};

// Block swap between two pools (device cache, host memory), per layer.
struct SwapParams {
    const void* src_k[kCopyMaxLayers];
    const void* src_v[kCopyMaxLayers];
    void* dst_k[kCopyMaxLayers];
    void* dst_v[kCopyMaxLayers];
    int32_t num_layers;
    int64_t src_blocks;
    int64_t dst_blocks;
    int64_t block_bytes;
    const int64_t* pairs;          // [num_pairs][2]: src block, dst block
    int64_t num_pairs;
    int32_t* dev_err;
};

cudaError_t launch_swap_blocks(const SwapParams& p, cudaStream_t stream);
// Streaming copy of `bytes` (a multiple of 16) with SM loads and stores.
cudaError_t launch_stream_copy(void* dst, const void* src, int64_t bytes, cudaStream_t stream);

// SHA-256 constants (FIPS 180-4 §4.2.2, §5.3.3), derived on the host.
struct Sha256Table {
    uint32_t k[64];
    uint32_t h0[8];
};

// Chained SHA-256 hashes of full blocks of token ids.
struct HashParams {
    const int32_t* token_ids;      // [total_tokens]
    const int32_t* cu_seqlens;     // [num_seqs + 1]
    int32_t num_seqs;
    int64_t total_tokens;
    int32_t block_size;
    const uint8_t* parent_hashes;  // [num_seqs][32] or null (zeros)
    const int64_t* block_offsets;  // [num_seqs]: index of each sequence's first hash
    int64_t total_blocks;          // rows of `hashes`
    uint8_t* hashes;               // [total_blocks][32]
    int32_t* dev_err;
    Sha256Table table;
};

cudaError_t launch_block_hashes(const HashParams& p, cudaStream_t stream);
const Sha256Table& sha256_table();

// Each returns cudaSuccess, or cudaErrorNotSupported for a shape without a kernel.
cudaError_t launch_decode_partitions(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode_stream(const DecodeParams& p, bool mma, cudaStream_t stream);
// Partials of the shared prefixes (p.grp_* set); NotSupported unless the cache
// and q are the same 16-bit type.
cudaError_t launch_decode_prefix(const DecodeParams& p, cudaStream_t stream);
bool prefix_kernel_supported(int cache_dtype, int q_dtype, int head_dim, int block_size,
                             int group);
// Single-pass shared-prefix decode (decode_group.cu): one CTA per (group, KV
// head, row tile) reads the shared blocks once and each member's own blocks,
// and writes out directly (no partials, no reduce).  Same shapes as the
// prefix kernel; NotSupported when the cache is too large for a tensor map.
cudaError_t launch_decode_group(const DecodeParams& p, cudaStream_t stream);
int64_t group_decode_ctas(const DecodeParams& p);
// Which shared-prefix path the calls take: 0 = the library's choice, 1 = the
// single pass, 2 = prefix kernel + partition kernel + reduce
// (pkv_testing_set_shared_prefix_path).
int32_t shared_prefix_path();
cudaError_t launch_lse_reduce(const ReduceParams& p, cudaStream_t stream, bool pdl);
cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_copy_blocks(const CopyParams& p, cudaStream_t stream);

// Which decode kernel a shape selects (for the host checks and tests).
bool decode_shape_supported(int cache_dtype, int q_dtype, int head_dim, int block_size);

}  // namespace pkv
