// pkv_api.cu -- the C ABI of include/pkv.h: argument checks, launch choice.
//
// Every entry point validates what the host can see (pointers, alignment,
// sizes, supported shapes) and returns before launching anything when a check
// fails.  Nothing here allocates, frees or synchronises.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

bool is16(int32_t dt) { return dt == PKV_F16 || dt == PKV_BF16; }

pkv_status check_cache(const pkv_cache_desc* c)
{
    if (c == nullptr || c->k_cache == nullptr || c->v_cache == nullptr)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(c->k_cache) || !aligned16(c->v_cache))
        return PKV_ERR_INVALID_ARG;
    if (c->num_blocks <= 0 || c->num_kv_heads <= 0 || c->block_size <= 0 || c->head_dim <= 0)
        return PKV_ERR_INVALID_ARG;
    if (c->cache_dtype != PKV_F16 && c->cache_dtype != PKV_BF16 && c->cache_dtype != PKV_FP8_E4M3)
        return PKV_ERR_INVALID_ARG;
    if (c->head_dim != 64 && c->head_dim != 128)
        return PKV_ERR_UNSUPPORTED;
    if (c->block_size != 8 && c->block_size != 16 && c->block_size != 32)
        return PKV_ERR_UNSUPPORTED;
    if (c->cache_dtype == PKV_FP8_E4M3) {
        if (!(c->k_scale > 0.f) || !(c->v_scale > 0.f) || c->k_scale != c->k_scale ||
            c->v_scale != c->v_scale)
            return PKV_ERR_INVALID_ARG;
    }
    return PKV_OK;
}

pkv_status from_cuda(cudaError_t e)
{
    if (e == cudaSuccess)
        return PKV_OK;
    if (e == cudaErrorNotSupported)
        return PKV_ERR_UNSUPPORTED;
    return PKV_ERR_CUDA;
}

struct WorkspaceLayout {
    int64_t parts;
    int64_t m_off, l_off, o_off, bytes;
};

// Partials per (sequence, head) row: ceil(max_context_len / partition_size),
// plus kPrefixParts when shared prefixes are cut into partitions of their own
// (at most kPrefixParts of them, then ceil((c - P) / ps) <= ceil(c / ps)).
WorkspaceLayout layout(int32_t num_seqs, int32_t num_heads, int32_t head_dim,
                       int32_t max_context_len, int32_t partition_size, bool prefixes = false)
{
    WorkspaceLayout w{};
    w.parts = partition_size > 0 ? ((int64_t)max_context_len + partition_size - 1) / partition_size
                                 : 0;
    if (prefixes && w.parts > 0)
        w.parts += pkv::kPrefixParts;
    if (w.parts <= 1) {
        w.bytes = 0;
        return w;
    }
    const int64_t rows = (int64_t)num_seqs * num_heads * w.parts;
    const int64_t ml = round_up(4 * rows, 256);
    w.m_off = 0;
    w.l_off = ml;
    w.o_off = 2 * ml;
    w.bytes = 2 * ml + round_up(4 * rows * head_dim, 256);
    return w;
}

// SM count of the current device, looked up once per device.
int device_sms()
{
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 152;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            v <= 0)
            return 152;
        cache[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

int32_t resolve_partition(const pkv_cache_desc* c, int32_t num_seqs, int32_t num_heads,
                          int32_t max_context_len, int32_t requested)
{
    if (requested > 0)
        return requested;
    const int32_t elem = c->cache_dtype == PKV_FP8_E4M3 ? 1 : 2;
    const int32_t group = c->num_kv_heads > 0 ? num_heads / c->num_kv_heads : 1;
    const bool grouped_items = group >= 2 && group <= 16 && c->cache_dtype != PKV_FP8_E4M3 &&
                               c->block_size % 16 == 0;
    // one partition per context when there are enough items to fill the GPU:
    // both kernels take the longest contexts first, which balances this many
    // items without a split (and the reduce launch disappears).  Items are
    // (sequence, query head) for the streaming kernel (persistent, 3 CTAs per
    // SM, 6 items per SM asked) and (sequence, KV head) for the grouped-head
    // kernel (one item per CTA, 3 resident per SM).  When the grouped items
    // fill one wave but not two, the longest contexts alone would run in the
    // tail, so contexts longer than 3/4 of the longest are cut in two.
    const int64_t items = grouped_items ? (int64_t)num_seqs * c->num_kv_heads
                                        : (int64_t)num_seqs * num_heads;
    const int64_t wave = 3 * (int64_t)device_sms();
    if (num_seqs > 0 && num_seqs <= 128 && max_context_len > 0 && max_context_len <= 8192) {
        const int32_t bs = c->block_size;
        if (items >= 2 * wave)
            return (max_context_len + bs - 1) / bs * bs;
        if (items >= wave) {
            if (!grouped_items)
                return (max_context_len + bs - 1) / bs * bs;
            const int32_t cut = (3 * max_context_len + 3) / 4;
            return (cut + bs - 1) / bs * bs;
        }
    }
    // K+V bytes of one KV head per partition: 256 KiB when a work item serves
    // one query head, 1 MiB when it serves a group of them
    const int64_t budget = grouped_items ? (1 << 20) : (1 << 18);
    int32_t tokens = (int32_t)(budget / (2 * c->head_dim * elem));
    tokens = tokens / c->block_size * c->block_size;
    return tokens < c->block_size ? c->block_size : tokens;
}

pkv_status decode_checks(const pkv_cache_desc* cache, const void* q, int32_t q_dtype,
                         int32_t num_seqs, int32_t num_heads, const int32_t* block_tables,
                         int32_t max_blocks_per_seq, const int32_t* context_lens,
                         int32_t max_context_len, int32_t partition_size, const void* out)
{
    pkv_status st = check_cache(cache);
    if (st != PKV_OK)
        return st;
    if (num_seqs < 0 || num_heads <= 0 || max_blocks_per_seq < 0 || max_context_len < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_heads % cache->num_kv_heads != 0)
        return PKV_ERR_INVALID_ARG;
    if (!is16(q_dtype))
        return PKV_ERR_INVALID_ARG;
    if (partition_size < 0 || (partition_size > 0 && partition_size % cache->block_size != 0))
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0)
        return PKV_OK;
    if (q == nullptr || out == nullptr || context_lens == nullptr || !aligned16(q) ||
        !aligned16(out))
        return PKV_ERR_INVALID_ARG;
    if (max_context_len > 0 && (block_tables == nullptr || max_blocks_per_seq <= 0))
        return PKV_ERR_INVALID_ARG;
    if (!pkv::decode_shape_supported(cache->cache_dtype, q_dtype, cache->head_dim,
                                     cache->block_size))
        return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

// Shared-prefix groups of one call (all zero for a plain decode).
struct Groups {
    const int32_t* begin;
    const int32_t* prefix_blocks;
    int32_t num;
    int32_t max_size;
    int32_t max_blocks;
    int32_t partition;     // prefix_partition
};

pkv::DecodeParams decode_params(const pkv_cache_desc* cache, const void* q, int32_t q_dtype,
                                int32_t num_seqs, int32_t num_heads,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* context_lens, int32_t max_context_len,
                                float scale, int32_t partition, void* workspace,
                                const WorkspaceLayout& wl, const Groups& grp, int32_t* dev_err,
                                void* out)
{
    pkv::DecodeParams p{};
    p.k_cache = cache->k_cache;
    p.v_cache = cache->v_cache;
    p.num_blocks = cache->num_blocks;
    p.num_kv_heads = cache->num_kv_heads;
    p.block_size = cache->block_size;
    p.head_dim = cache->head_dim;
    p.cache_dtype = cache->cache_dtype;
    const bool fp8 = cache->cache_dtype == PKV_FP8_E4M3;
    p.k_scale = fp8 ? cache->k_scale : 1.f;
    p.v_scale = fp8 ? cache->v_scale : 1.f;
    p.q = q;
    p.q_dtype = q_dtype;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.group = num_heads / cache->num_kv_heads;
    p.block_tables = block_tables;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.context_lens = context_lens;
    p.max_context_len = max_context_len;
    p.partition_size = partition;
    p.max_partitions = wl.parts < 1 ? 1 : (int32_t)wl.parts;
    p.grid_partitions = (int32_t)(((int64_t)max_context_len + partition - 1) / partition);
    if (p.grid_partitions < 1)
        p.grid_partitions = 1;
    p.qk_scale_log2 = scale * 1.4426950408889634f * p.k_scale;
    char* ws = reinterpret_cast<char*>(workspace);
    p.ws_m = wl.bytes ? reinterpret_cast<float*>(ws + wl.m_off) : nullptr;
    p.ws_l = wl.bytes ? reinterpret_cast<float*>(ws + wl.l_off) : nullptr;
    p.ws_o = wl.bytes ? reinterpret_cast<float*>(ws + wl.o_off) : nullptr;
    p.dev_err = dev_err;
    p.out = out;
    p.grp_begin = grp.begin;
    p.grp_prefix_blocks = grp.prefix_blocks;
    p.num_groups = grp.num;
    p.max_group_size = grp.max_size;
    p.max_prefix_blocks = grp.max_blocks;
    p.prefix_partition = grp.partition;
    p.wait_tries = pkv::decode_wait_tries();
    return p;
}

pkv_status launch_partitions(const pkv_cache_desc* cache, const void* q, int32_t q_dtype,
                             int32_t num_seqs, int32_t num_heads, const int32_t* block_tables,
                             int32_t max_blocks_per_seq, const int32_t* context_lens,
                             int32_t max_context_len, float scale, int32_t partition,
                             void* workspace, const WorkspaceLayout& wl, int32_t* dev_err,
                             void* out, cudaStream_t stream, const Groups& grp = Groups{})
{
    const pkv::DecodeParams p =
        decode_params(cache, q, q_dtype, num_seqs, num_heads, block_tables, max_blocks_per_seq,
                      context_lens, max_context_len, scale, partition, workspace, wl, grp,
                      dev_err, out);
    return from_cuda(pkv::launch_decode_partitions(p, stream));
}

pkv_status launch_reduce(int32_t num_seqs, int32_t num_heads, int32_t head_dim,
                         const int32_t* context_lens, int32_t max_context_len, int32_t partition,
                         const void* workspace, const WorkspaceLayout& wl, int32_t out_dtype,
                         void* out, cudaStream_t stream, bool pdl, int32_t block_size = 0,
                         const Groups& grp = Groups{})
{
    if (wl.bytes == 0)
        return PKV_OK;
    pkv::ReduceParams r{};
    r.num_seqs = num_seqs;
    r.num_heads = num_heads;
    r.head_dim = head_dim;
    r.context_lens = context_lens;
    r.max_context_len = max_context_len;
    r.partition_size = partition;
    r.max_partitions = (int32_t)wl.parts;
    const char* ws = reinterpret_cast<const char*>(workspace);
    r.ws_m = reinterpret_cast<const float*>(ws + wl.m_off);
    r.ws_l = reinterpret_cast<const float*>(ws + wl.l_off);
    r.ws_o = reinterpret_cast<const float*>(ws + wl.o_off);
    r.out_dtype = out_dtype;
    r.out = out;
    r.block_size = block_size;
    r.grp_begin = grp.begin;
    r.grp_prefix_blocks = grp.prefix_blocks;
    r.num_groups = grp.num;
    r.max_group_size = grp.max_size;
    r.max_prefix_blocks = grp.max_blocks;
    r.prefix_partition = grp.partition;
    return from_cuda(pkv::launch_lse_reduce(r, stream, pdl));
}

// A pointer the GPU can dereference: device memory, or host memory that is
// pinned and mapped into the device's address space (its device address is
// returned; with unified addressing it is the same pointer).
bool device_reachable(const void* p, void** dev_ptr)
{
    cudaPointerAttributes a{};
    if (p == nullptr || cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged ||
        a.type == cudaMemoryTypeHost) {
        if (a.devicePointer == nullptr)
            return false;
        *dev_ptr = a.devicePointer;
        return true;
    }
    return false;
}

pkv_status check_workspace(const WorkspaceLayout& wl, const void* workspace, size_t bytes)
{
    if (wl.bytes == 0)
        return PKV_OK;
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return PKV_ERR_WORKSPACE;
    if ((int64_t)bytes < wl.bytes)
        return PKV_ERR_WORKSPACE;
    return PKV_OK;
}

// The wait limit that pkv_testing_set_decode_wait_limit sets (0 = the
// kernels' own).
std::atomic<uint32_t> g_decode_wait_tries{0};
// The shared-prefix path that pkv_testing_set_shared_prefix_path sets.
std::atomic<int32_t> g_shared_prefix_path{0};

// Longest context the single-pass shared-prefix decode takes by itself: one
// CTA streams the prefix and every member's own blocks of its row tile, so
// its work grows with the contexts; beyond this the split path balances
// better.
constexpr int32_t kGroupMaxContext = 4096;

}  // namespace

uint32_t pkv::decode_wait_tries()
{
    return g_decode_wait_tries.load(std::memory_order_relaxed);
}

int32_t pkv::shared_prefix_path()
{
    return g_shared_prefix_path.load(std::memory_order_relaxed);
}

extern "C" {

uint32_t pkv_testing_set_decode_wait_limit(uint32_t tries)
{
    return g_decode_wait_tries.exchange(tries, std::memory_order_relaxed);
}

int32_t pkv_testing_set_shared_prefix_path(int32_t path)
{
    if (path < 0 || path > 2)
        return -1;
    return g_shared_prefix_path.exchange(path, std::memory_order_relaxed);
}


const char* pkv_status_string(int32_t status)
{
    switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape or type";
    case PKV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case PKV_ERR_CUDA: return "CUDA launch failed";
    case PKV_ERR_SCRATCH_LIMIT:
        return "request exceeds the library's static decode scratch (PKV_STATIC_SCRATCH_BYTES)";
    default: return "unknown status";
    }
}

pkv_status pkv_kv_append(const pkv_cache_desc* cache, const void* k, const void* v,
                         int32_t in_dtype, const int64_t* slot_mapping, int64_t num_tokens,
                         int32_t* dev_err, pkv_stream_t stream)
{
    pkv_status st = check_cache(cache);
    if (st != PKV_OK)
        return st;
    if (num_tokens < 0 || !is16(in_dtype))
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0)
        return PKV_OK;
    if (k == nullptr || v == nullptr || slot_mapping == nullptr || !aligned16(k) || !aligned16(v))
        return PKV_ERR_INVALID_ARG;
    if (cache->cache_dtype != in_dtype && cache->cache_dtype != PKV_FP8_E4M3)
        return PKV_ERR_UNSUPPORTED;
    pkv::AppendParams p{};
    p.k_cache = cache->k_cache;
    p.v_cache = cache->v_cache;
    p.num_blocks = cache->num_blocks;
    p.num_kv_heads = cache->num_kv_heads;
    p.block_size = cache->block_size;
    p.head_dim = cache->head_dim;
    p.cache_dtype = cache->cache_dtype;
    p.k_inv_scale = cache->cache_dtype == PKV_FP8_E4M3 ? 1.0f / cache->k_scale : 1.f;
    p.v_inv_scale = cache->cache_dtype == PKV_FP8_E4M3 ? 1.0f / cache->v_scale : 1.f;
    p.k = k;
    p.v = v;
    p.in_dtype = in_dtype;
    p.slot_mapping = slot_mapping;
    p.num_tokens = num_tokens;
    p.dev_err = dev_err;
    return from_cuda(pkv::launch_kv_append(p, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_copy_blocks(const pkv_cache_desc* caches, int32_t num_layers,
                           const int64_t* block_pairs, int64_t num_pairs, int32_t* dev_err,
                           pkv_stream_t stream)
{
    if (caches == nullptr || num_layers <= 0 || num_pairs < 0)
        return PKV_ERR_INVALID_ARG;
    for (int32_t l = 0; l < num_layers; ++l) {
        pkv_status st = check_cache(&caches[l]);
        if (st != PKV_OK)
            return st;
        const pkv_cache_desc& a = caches[0];
        const pkv_cache_desc& b = caches[l];
        if (a.num_blocks != b.num_blocks || a.num_kv_heads != b.num_kv_heads ||
            a.block_size != b.block_size || a.head_dim != b.head_dim ||
            a.cache_dtype != b.cache_dtype)
            return PKV_ERR_INVALID_ARG;
    }
    if (num_pairs == 0)
        return PKV_OK;
    if (block_pairs == nullptr)
        return PKV_ERR_INVALID_ARG;
    const pkv_cache_desc& c0 = caches[0];
    const int64_t elem = c0.cache_dtype == PKV_FP8_E4M3 ? 1 : 2;
    pkv::CopyParams p{};
    p.num_blocks = c0.num_blocks;
    p.block_bytes = (int64_t)c0.num_kv_heads * c0.block_size * c0.head_dim * elem;
    p.dev_err = dev_err;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (int32_t l0 = 0; l0 < num_layers; l0 += pkv::kCopyMaxLayers) {
        const int32_t nl = num_layers - l0 < pkv::kCopyMaxLayers ? num_layers - l0
                                                                 : pkv::kCopyMaxLayers;
        p.num_layers = nl;
        for (int32_t i = 0; i < nl; ++i) {
            p.k[i] = caches[l0 + i].k_cache;
            p.v[i] = caches[l0 + i].v_cache;
        }
        for (int64_t q0 = 0; q0 < num_pairs; q0 += 65535) {
            p.pairs = block_pairs + 2 * q0;
            p.num_pairs = num_pairs - q0 < 65535 ? num_pairs - q0 : 65535;
            pkv_status st = from_cuda(pkv::launch_copy_blocks(p, s));
            if (st != PKV_OK)
                return st;
        }
    }
    return PKV_OK;
}

int32_t pkv_decode_partition_size(const pkv_cache_desc* cache, int32_t num_seqs,
                                  int32_t num_heads, int32_t max_context_len, int32_t requested)
{
    if (cache == nullptr || cache->block_size <= 0 || cache->head_dim <= 0)
        return 0;
    return resolve_partition(cache, num_seqs, num_heads, max_context_len, requested);
}

size_t pkv_decode_workspace_bytes(const pkv_cache_desc* cache, int32_t num_seqs,
                                  int32_t num_heads, int32_t max_context_len,
                                  int32_t partition_size)
{
    if (cache == nullptr || cache->block_size <= 0 || cache->head_dim <= 0 || num_seqs <= 0 ||
        num_heads <= 0 || max_context_len <= 0 || partition_size < 0)
        return 0;
    const int32_t part = resolve_partition(cache, num_seqs, num_heads, max_context_len,
                                           partition_size);
    return (size_t)layout(num_seqs, num_heads, cache->head_dim, max_context_len, part).bytes;
}

pkv_status pkv_paged_attention_partitions(const pkv_cache_desc* cache, const void* q,
                                          int32_t q_dtype, int32_t num_seqs, int32_t num_heads,
                                          const int32_t* block_tables,
                                          int32_t max_blocks_per_seq,
                                          const int32_t* context_lens, int32_t max_context_len,
                                          float scale, int32_t partition_size, void* workspace,
                                          size_t workspace_bytes, int32_t* dev_err, void* out,
                                          pkv_stream_t stream)
{
    pkv_status st = decode_checks(cache, q, q_dtype, num_seqs, num_heads, block_tables,
                                  max_blocks_per_seq, context_lens, max_context_len,
                                  partition_size, out);
    if (st != PKV_OK || num_seqs == 0)
        return st;
    const int32_t part = resolve_partition(cache, num_seqs, num_heads, max_context_len,
                                           partition_size);
    const WorkspaceLayout wl = layout(num_seqs, num_heads, cache->head_dim, max_context_len, part);
    st = check_workspace(wl, workspace, workspace_bytes);
    if (st != PKV_OK)
        return st;
    return launch_partitions(cache, q, q_dtype, num_seqs, num_heads, block_tables,
                             max_blocks_per_seq, context_lens, max_context_len, scale, part,
                             workspace, wl, dev_err, out, reinterpret_cast<cudaStream_t>(stream));
}

pkv_status pkv_lse_reduce(int32_t num_seqs, int32_t num_heads, int32_t head_dim,
                          const int32_t* context_lens, int32_t max_context_len,
                          int32_t partition_size, const void* workspace, size_t workspace_bytes,
                          int32_t out_dtype, void* out, pkv_stream_t stream)
{
    if (num_seqs < 0 || num_heads <= 0 || max_context_len < 0 || partition_size <= 0 ||
        (head_dim != 64 && head_dim != 128) || !is16(out_dtype))
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0)
        return PKV_OK;
    if (context_lens == nullptr || out == nullptr || !aligned16(out))
        return PKV_ERR_INVALID_ARG;
    const WorkspaceLayout wl = layout(num_seqs, num_heads, head_dim, max_context_len,
                                      partition_size);
    pkv_status st = check_workspace(wl, workspace, workspace_bytes);
    if (st != PKV_OK)
        return st;
    return launch_reduce(num_seqs, num_heads, head_dim, context_lens, max_context_len,
                         partition_size, workspace, wl, out_dtype, out,
                         reinterpret_cast<cudaStream_t>(stream), false);
}

pkv_status pkv_paged_attention_decode(const pkv_cache_desc* cache, const void* q, int32_t q_dtype,
                                      int32_t num_seqs, int32_t num_heads,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* context_lens, int32_t max_context_len,
                                      float scale, int32_t partition_size, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_err, void* out,
                                      pkv_stream_t stream)
{
    pkv_status st = decode_checks(cache, q, q_dtype, num_seqs, num_heads, block_tables,
                                  max_blocks_per_seq, context_lens, max_context_len,
                                  partition_size, out);
    if (st != PKV_OK || num_seqs == 0)
        return st;
    const int32_t part = resolve_partition(cache, num_seqs, num_heads, max_context_len,
                                           partition_size);
    const WorkspaceLayout wl = layout(num_seqs, num_heads, cache->head_dim, max_context_len, part);
    st = check_workspace(wl, workspace, workspace_bytes);
    if (st != PKV_OK)
        return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    st = launch_partitions(cache, q, q_dtype, num_seqs, num_heads, block_tables,
                           max_blocks_per_seq, context_lens, max_context_len, scale, part,
                           workspace, wl, dev_err, out, s);
    if (st != PKV_OK)
        return st;
    return launch_reduce(num_seqs, num_heads, cache->head_dim, context_lens, max_context_len,
                         part, workspace, wl, q_dtype, out, s, true);
}

size_t pkv_shared_prefix_workspace_bytes(const pkv_cache_desc* cache, int32_t num_seqs,
                                         int32_t num_heads, int32_t max_context_len,
                                         int32_t partition_size)
{
    if (cache == nullptr || cache->block_size <= 0 || cache->head_dim <= 0 || num_seqs <= 0 ||
        num_heads <= 0 || max_context_len <= 0 || partition_size < 0)
        return 0;
    const int32_t part = resolve_partition(cache, num_seqs, num_heads, max_context_len,
                                           partition_size);
    return (size_t)layout(num_seqs, num_heads, cache->head_dim, max_context_len, part, true).bytes;
}

pkv_status pkv_paged_attention_decode_shared_prefix(
    const pkv_cache_desc* cache, const void* q, int32_t q_dtype, int32_t num_seqs,
    int32_t num_heads, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* context_lens, int32_t max_context_len, int32_t num_groups,
    const int32_t* group_begin, const int32_t* group_prefix_blocks, int32_t max_group_size,
    int32_t max_prefix_blocks, float scale, int32_t partition_size, void* workspace,
    size_t workspace_bytes, int32_t* dev_err, void* out, pkv_stream_t stream)
{
    pkv_status st = decode_checks(cache, q, q_dtype, num_seqs, num_heads, block_tables,
                                  max_blocks_per_seq, context_lens, max_context_len,
                                  partition_size, out);
    if (st != PKV_OK || num_seqs == 0)
        return st;
    if (num_groups < 0 || max_group_size < 0 || max_prefix_blocks < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_groups > 0 && (group_begin == nullptr || group_prefix_blocks == nullptr ||
                           max_group_size == 0 || num_groups > num_seqs))
        return PKV_ERR_INVALID_ARG;
    if ((int64_t)max_prefix_blocks * cache->block_size > max_context_len ||
        max_prefix_blocks > max_blocks_per_seq)
        return PKV_ERR_INVALID_ARG;
    if (!pkv::prefix_kernel_supported(cache->cache_dtype, q_dtype, cache->head_dim,
                                      cache->block_size, num_heads / cache->num_kv_heads))
        return PKV_ERR_UNSUPPORTED;
    const int32_t part = resolve_partition(cache, num_seqs, num_heads, max_context_len,
                                           partition_size);
    Groups grp{};
    if (num_groups > 0 && max_prefix_blocks > 0) {
        const int32_t bs = cache->block_size;
        const int32_t tokens = max_prefix_blocks * bs;
        const int32_t per = (tokens + pkv::kPrefixParts - 1) / pkv::kPrefixParts;
        const int32_t piece = (per + bs - 1) / bs * bs;
        grp = Groups{group_begin, group_prefix_blocks, num_groups, max_group_size,
                     max_prefix_blocks, piece > part ? piece : part};
    }
    const bool prefixes = grp.num > 0;
    const WorkspaceLayout wl =
        layout(num_seqs, num_heads, cache->head_dim, max_context_len, part, prefixes);
    st = check_workspace(wl, workspace, workspace_bytes);
    if (st != PKV_OK)
        return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (prefixes) {
        // Single pass (one CTA per group, KV head and row tile; no partials)
        // when the library chooses the split (partition_size 0), the contexts
        // are short enough for one CTA to stream a tile's members, and the
        // CTAs cover the GPU at least once.
        const pkv::DecodeParams p =
            decode_params(cache, q, q_dtype, num_seqs, num_heads, block_tables,
                          max_blocks_per_seq, context_lens, max_context_len, scale, part,
                          workspace, wl, grp, dev_err, out);
        const int32_t path = pkv::shared_prefix_path();
        const bool single = path == 1 ||
                            (path == 0 && partition_size == 0 &&
                             max_context_len <= kGroupMaxContext &&
                             pkv::group_decode_ctas(p) >= device_sms());
        if (single) {
            const cudaError_t e = pkv::launch_decode_group(p, s);
            if (e != cudaErrorNotSupported)
                return from_cuda(e);
        }
    }
    if (prefixes) {
        const pkv::DecodeParams p =
            decode_params(cache, q, q_dtype, num_seqs, num_heads, block_tables,
                          max_blocks_per_seq, context_lens, max_context_len, scale, part,
                          workspace, wl, grp, dev_err, out);
        st = from_cuda(pkv::launch_decode_prefix(p, s));
        if (st != PKV_OK)
            return st;
    }
    {
        // the partition kernel overlaps the prefix kernel (it reads nothing the
        // prefix kernel writes) and waits for it only before it exits
        pkv::DecodeParams p =
            decode_params(cache, q, q_dtype, num_seqs, num_heads, block_tables,
                          max_blocks_per_seq, context_lens, max_context_len, scale, part,
                          workspace, wl, grp, dev_err, out);
        p.wait_prior = prefixes ? 1 : 0;
        st = from_cuda(pkv::launch_decode_partitions(p, s));
        if (st != PKV_OK)
            return st;
    }
    return launch_reduce(num_seqs, num_heads, cache->head_dim, context_lens, max_context_len,
                         part, workspace, wl, q_dtype, out, s, true, cache->block_size, grp);
}

pkv_status pkv_paged_attention_prefill(const pkv_cache_desc* cache, const void* q,
                                       int32_t q_dtype, int32_t num_seqs, int32_t num_heads,
                                       const int32_t* cu_seqlens_q, int32_t total_q,
                                       int32_t max_q_len, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* context_lens,
                                       int32_t max_context_len, float scale, int32_t* dev_err,
                                       void* out, pkv_stream_t stream)
{
    pkv_status st = check_cache(cache);
    if (st != PKV_OK)
        return st;
    if (num_seqs < 0 || num_heads <= 0 || total_q < 0 || max_q_len < 0 ||
        max_blocks_per_seq < 0 || max_context_len < 0 || !is16(q_dtype))
        return PKV_ERR_INVALID_ARG;
    if (num_heads % cache->num_kv_heads != 0)
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0 || total_q == 0 || max_q_len == 0)
        return PKV_OK;
    if (q == nullptr || out == nullptr || cu_seqlens_q == nullptr || context_lens == nullptr ||
        block_tables == nullptr || max_blocks_per_seq == 0 || !aligned16(q) || !aligned16(out))
        return PKV_ERR_INVALID_ARG;
    if (!pkv::prefill_shape_supported(cache->cache_dtype, cache->head_dim, cache->block_size,
                                      num_heads / cache->num_kv_heads) ||
        q_dtype != cache->cache_dtype)
        return PKV_ERR_UNSUPPORTED;
    pkv::PrefillParams p{};
    p.k_cache = cache->k_cache;
    p.v_cache = cache->v_cache;
    p.num_blocks = cache->num_blocks;
    p.num_kv_heads = cache->num_kv_heads;
    p.block_size = cache->block_size;
    p.head_dim = cache->head_dim;
    p.dtype = cache->cache_dtype;
    p.q = q;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.group = num_heads / cache->num_kv_heads;
    p.cu_seqlens_q = cu_seqlens_q;
    p.total_q = total_q;
    p.max_q_len = max_q_len;
    p.block_tables = block_tables;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.context_lens = context_lens;
    p.max_context_len = max_context_len;
    p.qk_scale_log2 = scale * 1.4426950408889634f;
    p.dev_err = dev_err;
    p.out = out;
    return from_cuda(pkv::launch_prefill(p, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_swap_blocks(const pkv_cache_desc* src, const pkv_cache_desc* dst,
                           int32_t num_layers, const int64_t* block_pairs, int64_t num_pairs,
                           int32_t* dev_err, pkv_stream_t stream)
{
    if (src == nullptr || dst == nullptr || num_layers <= 0 || num_pairs < 0)
        return PKV_ERR_INVALID_ARG;
    for (int32_t l = 0; l < num_layers; ++l) {
        pkv_status st = check_cache(&src[l]);
        if (st == PKV_OK)
            st = check_cache(&dst[l]);
        if (st != PKV_OK)
            return st;
        const pkv_cache_desc& a = src[l];
        const pkv_cache_desc& b = dst[l];
        if (a.num_kv_heads != b.num_kv_heads || a.block_size != b.block_size ||
            a.head_dim != b.head_dim || a.cache_dtype != b.cache_dtype ||
            a.num_blocks != src[0].num_blocks || b.num_blocks != dst[0].num_blocks ||
            a.num_kv_heads != src[0].num_kv_heads || a.block_size != src[0].block_size ||
            a.head_dim != src[0].head_dim || a.cache_dtype != src[0].cache_dtype)
            return PKV_ERR_INVALID_ARG;
    }
    if (num_pairs == 0)
        return PKV_OK;
    void* pairs_dev = nullptr;
    if (!device_reachable(block_pairs, &pairs_dev))
        return PKV_ERR_INVALID_ARG;
    const pkv_cache_desc& c0 = src[0];
    const int64_t elem = c0.cache_dtype == PKV_FP8_E4M3 ? 1 : 2;
    pkv::SwapParams p{};
    p.src_blocks = src[0].num_blocks;
    p.dst_blocks = dst[0].num_blocks;
    p.block_bytes = (int64_t)c0.num_kv_heads * c0.block_size * c0.head_dim * elem;
    p.dev_err = dev_err;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (int32_t l0 = 0; l0 < num_layers; l0 += pkv::kCopyMaxLayers) {
        const int32_t nl = num_layers - l0 < pkv::kCopyMaxLayers ? num_layers - l0
                                                                 : pkv::kCopyMaxLayers;
        p.num_layers = nl;
        for (int32_t i = 0; i < nl; ++i) {
            void* ptrs[4];
            if (!device_reachable(src[l0 + i].k_cache, &ptrs[0]) ||
                !device_reachable(src[l0 + i].v_cache, &ptrs[1]) ||
                !device_reachable(dst[l0 + i].k_cache, &ptrs[2]) ||
                !device_reachable(dst[l0 + i].v_cache, &ptrs[3]))
                return PKV_ERR_INVALID_ARG;
            p.src_k[i] = ptrs[0];
            p.src_v[i] = ptrs[1];
            p.dst_k[i] = ptrs[2];
            p.dst_v[i] = ptrs[3];
        }
        for (int64_t q0 = 0; q0 < num_pairs; q0 += 65535) {
            p.pairs = reinterpret_cast<const int64_t*>(pairs_dev) + 2 * q0;
            p.num_pairs = num_pairs - q0 < 65535 ? num_pairs - q0 : 65535;
            pkv_status st = from_cuda(pkv::launch_swap_blocks(p, s));
            if (st != PKV_OK)
                return st;
        }
    }
    return PKV_OK;
}

pkv_status pkv_testing_stream_copy(void* dst, const void* src, int64_t bytes,
                                   pkv_stream_t stream)
{
    if (bytes < 0 || bytes % 16 != 0 || !aligned16(dst) || !aligned16(src))
        return PKV_ERR_INVALID_ARG;
    if (bytes == 0)
        return PKV_OK;
    void* d = nullptr;
    void* s = nullptr;
    if (!device_reachable(dst, &d) || !device_reachable(src, &s))
        return PKV_ERR_INVALID_ARG;
    return from_cuda(pkv::launch_stream_copy(d, s, bytes, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_block_hashes(const int32_t* token_ids, const int32_t* cu_seqlens,
                            int32_t num_seqs, int64_t total_tokens, int32_t block_size,
                            const uint8_t* parent_hashes, const int64_t* block_offsets,
                            int64_t total_blocks, uint8_t* hashes, int32_t* dev_err,
                            pkv_stream_t stream)
{
    if (num_seqs < 0 || total_tokens < 0 || total_blocks < 0)
        return PKV_ERR_INVALID_ARG;
    if (block_size != 8 && block_size != 16 && block_size != 32)
        return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0)
        return PKV_OK;
    if (cu_seqlens == nullptr || block_offsets == nullptr ||
        (total_tokens > 0 && token_ids == nullptr) || (total_blocks > 0 && hashes == nullptr) ||
        !aligned16(hashes) || !aligned16(parent_hashes))
        return PKV_ERR_INVALID_ARG;
    pkv::HashParams p{};
    p.token_ids = token_ids;
    p.cu_seqlens = cu_seqlens;
    p.num_seqs = num_seqs;
    p.total_tokens = total_tokens;
    p.block_size = block_size;
    p.parent_hashes = parent_hashes;
    p.block_offsets = block_offsets;
    p.total_blocks = total_blocks;
    p.hashes = hashes;
    p.dev_err = dev_err;
    p.table = pkv::sha256_table();
    return from_cuda(pkv::launch_block_hashes(p, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
