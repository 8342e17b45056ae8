/*
 * pkv.h -- C ABI of the paged KV-cache decode library (libpkv.so, sm_103a).
 *
 * The library implements the data-parallel hot path of PagedAttention: the
 * per-token append of K/V into a cache of fixed-size physical blocks, the
 * copy-on-write block copy, and single-query decode attention that walks each
 * sequence's block table.  The operations are those of the pages
 *   「KV 缓存与分页注意力」 (Laplace mini-world plate F55): §02 一次写一个词元
 *   (each decode round computes and stores only the new token's K/V, then
 *   attends over all earlier K/V), §06 像内存分页 (equal-size blocks, logical
 *   vs physical), §07 块表 (block table; the kernel fetches K/V block by block
 *   through it), §08 共用，写时复制 (shared blocks, copy before writing), §11
 *   后来的做法 (query heads in groups sharing one K/V head; 8-bit float cache);
 *   「Paged Attention in LLMs」 (Outcome School, Chinese translation), sections
 *   "Paged Attention 如何工作" and "Block Table".
 *
 * Conventions shared by every call
 * --------------------------------
 * Ownership.  The caller owns every buffer.  The library never allocates,
 *   frees or synchronises, and it is thread-safe.  A pkv_cache_desc holds
 *   raw pointers and no reference: the caches it names must stay allocated
 *   (and mapped) for as long as any call that uses the descriptor may run,
 *   including every replay of a CUDA graph that captured such a call.  Between calls it keeps only
 *   a per-device record of each decode kernel's launch size and a static
 *   device table of work counters for the streaming decode kernel (the
 *   single-head and FP8 decode): 1024 slots, each reset to zero by the last
 *   CTA of the launch that used it.  A launch takes the next slot in turn
 *   when it is issued, or captured into a CUDA graph (a graph keeps its slot
 *   for every replay).  Two launches may therefore share a slot only if they
 *   run at the same time: more than 1024 decode launches in flight at once,
 *   or one captured decode graph replayed on two streams at once, or replayed
 *   while the direct decode launch issued 1024 launches after its capture
 *   (which takes the same slot) still runs on another stream.  Avoid those;
 *   launches on one stream, and graph replays on one stream, never share a
 *   slot.  A shared slot makes work items be skipped; the kernels then set
 *   PKV_DEVERR_SCHED when they see it (more claims or finished CTAs than one
 *   launch can make), though an overlap can go unseen.
 * Pointers.   "device" pointers must be CUDA device (or managed) memory of
 *   the current device.  Element data (caches, q, k, v, out) must be 16-byte
 *   aligned and dense row-major in the shapes given.
 * Execution.  Every compute call is asynchronous on `stream` (NULL = the
 *   legacy default stream).  Errors that the host can see (bad sizes, null or
 *   misaligned pointers, unsupported shapes) return before anything is
 *   launched.  A failed launch returns PKV_ERR_CUDA.
 * Device-side checks.  Every index read from device memory (slot, block id,
 *   context length, copy pair) is range-checked inside the kernels; an access
 *   that would leave its buffer is skipped, never performed.  When `dev_err`
 *   is non-NULL the kernel ORs the PKV_DEVERR_* bits of what it found into
 *   that device int32 (the caller zeroes it and reads it back).
 * Element types.  PKV_F16 (IEEE binary16), PKV_BF16, PKV_FP8_E4M3 (OCP E4M3,
 *   the "fn" variant: no infinities, largest finite 448).
 * Cache layout.  One layer's K cache and V cache are separate arrays of shape
 *   [num_blocks][num_kv_heads][block_size][head_dim]; the slot of a token is
 *   block * block_size + offset.  A (block, KV head) tile is therefore one
 *   contiguous run of block_size * head_dim elements.
 * Supported shapes.  head_dim in {64, 128}; block_size in {8, 16, 32};
 *   num_heads a multiple of num_kv_heads.  A 16-bit cache is read with a q of
 *   the same type; an FP8 cache with an fp16 or bf16 q.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (the same handle as cudaStream_t / CUstream). */
typedef struct CUstream_st* pkv_stream_t;

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or count  */
    PKV_ERR_UNSUPPORTED = 2,   /* shape or type combination not implemented   */
    PKV_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required  */
    PKV_ERR_CUDA = 4,          /* a kernel launch failed                      */
    PKV_ERR_SCRATCH_LIMIT = 5  /* request exceeds the static decode scratch   */
} pkv_status;

typedef enum pkv_dtype {
    PKV_F16 = 0,
    PKV_BF16 = 1,
    PKV_FP8_E4M3 = 2
} pkv_dtype;

/* Bits a kernel ORs into *dev_err. */
#define PKV_DEVERR_SLOT      1   /* slot >= num_blocks * block_size            */
#define PKV_DEVERR_BLOCK_ID  2   /* block-table entry outside [0, num_blocks)  */
#define PKV_DEVERR_CONTEXT   4   /* context length < 0, above max_context_len  */
                                 /* or above max_blocks_per_seq * block_size   */
#define PKV_DEVERR_COPY_PAIR 8   /* copy pair entry outside [0, num_blocks)    */
#define PKV_DEVERR_TIMEOUT   16  /* a kernel's bounded wait on its own copies  */
                                 /* ran out; that call's output is not valid   */
#define PKV_DEVERR_PREFIX    32  /* a shared-prefix group entry is unusable, or */
                                 /* a member's table differs within the prefix */
#define PKV_DEVERR_SCHED     64  /* a decode launch found its work-counter slot */
                                 /* in use by another launch in flight; that   */
                                 /* call's output is not valid (see Ownership) */

/* One layer's cache.  k_cache / v_cache: device, caller-owned, layout above.
 * k_scale / v_scale: for an FP8 cache, the stored code times the scale is the
 * value (one fp32 scale per tensor); ignored (treated as 1) otherwise. */
typedef struct pkv_cache_desc {
    void* k_cache;
    void* v_cache;
    int64_t num_blocks;
    int32_t num_kv_heads;
    int32_t block_size;
    int32_t head_dim;
    int32_t cache_dtype;          /* pkv_dtype */
    float k_scale;
    float v_scale;
} pkv_cache_desc;

/* Human-readable name of a status code (static string). */
const char* pkv_status_string(int32_t status);

/* ---------------------------------------------------------------------------
 * kv_append -- write each new token's K and V into its slot.
 *   「KV 缓存与分页注意力」 §02 (the new token's K/V are computed once and kept)
 *   and §07 (the slot comes from the sequence's block table).
 *
 * k, v          device [num_tokens][num_kv_heads][head_dim] of in_dtype
 *               (PKV_F16 or PKV_BF16).
 * slot_mapping  device int64 [num_tokens]; token t goes to block
 *               slot / block_size, offset slot % block_size, every KV head.
 *               A negative slot skips the token (padding).  A slot at or past
 *               num_blocks * block_size is skipped and flagged.
 * Result: with a cache of in_dtype the bytes are copied unchanged.  With an
 *   FP8 cache each element is stored as E4M3(fp32(x) * (1.0f / scale)), round
 *   to nearest even, saturating to +-448, scale = k_scale or v_scale.
 *   Other type pairings return PKV_ERR_UNSUPPORTED.
 * Precondition (not checked): the non-negative slots are distinct.
 * num_tokens == 0 is a no-op.
 * ------------------------------------------------------------------------- */
pkv_status pkv_kv_append(const pkv_cache_desc* cache,
                         const void* k, const void* v, int32_t in_dtype,
                         const int64_t* slot_mapping, int64_t num_tokens,
                         int32_t* dev_err, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * copy_blocks -- copy-on-write block copy.
 *   「KV 缓存与分页注意力」 §08 (before writing into a block that other
 *   sequences share, the writer copies the block and writes into the copy).
 *
 * caches      host array of num_layers descriptors, all with the same
 *             num_blocks / num_kv_heads / block_size / head_dim / cache_dtype.
 * block_pairs device int64 [num_pairs][2] = (src, dst) physical block ids.
 * Result: for every layer and pair, the whole dst block of K and of V (all
 *   heads, all block_size slots) becomes a copy of the src block.  A pair with
 *   an id outside [0, num_blocks) is skipped and flagged.
 * Precondition (not checked): dst ids are distinct and no dst is also a src.
 * num_pairs == 0 is a no-op.
 * ------------------------------------------------------------------------- */
pkv_status pkv_copy_blocks(const pkv_cache_desc* caches, int32_t num_layers,
                           const int64_t* block_pairs, int64_t num_pairs,
                           int32_t* dev_err, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * Block swap -- move whole blocks between two pools, typically the device
 * cache and a pool in pinned host memory: a pre-empted sequence's blocks go to
 * CPU memory and come back when it runs again (「KV 缓存与分页注意力」 §09).
 *
 * For each pair i and each layer l:
 *   dst[l].k_cache[pairs[i][1]] = src[l].k_cache[pairs[i][0]]  (and v_cache)
 * byte for byte; a block is num_kv_heads * block_size * head_dim elements.
 * src, dst        host arrays of num_layers descriptors; every layer of a side
 *                 has the same shape and pool size, and both sides the same
 *                 block shape and element type.  Each cache pointer must be
 *                 device memory or pinned, device-mapped host memory (checked
 *                 with cudaPointerGetAttributes; anything else returns
 *                 PKV_ERR_INVALID_ARG before any launch).  On GB300 the kernel
 *                 reads and writes the host side directly over NVLink-C2C.
 * block_pairs     int64 [num_pairs][2] (src block, dst block), device or
 *                 pinned host memory; dst blocks must be distinct.
 * A pair outside its pool is skipped and flags PKV_DEVERR_COPY_PAIR.
 * Launches: one kernel per 64 layers and 65,535 pairs.
 * ------------------------------------------------------------------------- */
pkv_status pkv_swap_blocks(const pkv_cache_desc* src, const pkv_cache_desc* dst,
                           int32_t num_layers, const int64_t* block_pairs, int64_t num_pairs,
                           int32_t* dev_err, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_testing_stream_copy -- a measurement aid, not part of the method (the
 * pages have no counterpart).
 *
 * Copies `bytes` (a multiple of 16) from src to dst with plain SM loads and
 * stores, many 16-byte vectors in flight per thread, as a reference for what
 * a copy kernel can reach over a given link: between device memory and
 * pinned, device-mapped host memory it shows the NVLink-C2C rate that SMs
 * see, which pkv_swap_blocks is measured against (the copy engines'
 * cudaMemcpyAsync rate is a different path).  Both pointers must be 16-byte
 * aligned and reachable by the GPU (device memory, or pinned host memory;
 * checked with cudaPointerGetAttributes, else PKV_ERR_INVALID_ARG before any
 * launch).  The ranges must not overlap.  Asynchronous on `stream`.
 * ------------------------------------------------------------------------- */
pkv_status pkv_testing_stream_copy(void* dst, const void* src, int64_t bytes,
                                   pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * Block hashes for prefix caching -- every full block gets a hash of its
 * tokens and of all the content in front of it, so that requests with the same
 * opening find the same blocks (「KV 缓存与分页注意力」 §11; 「KV Cache从原理到实战」
 * §4.2).  The hash function is this library's choice (the pages name none):
 *   h_i = SHA-256(h_{i-1} || token ids of block i as little-endian int32)
 * (FIPS 180-4), with h_{-1} = parent_hashes[s] or 32 zero bytes.  A partial
 * last block gets no hash.
 *
 * token_ids      device int32 [total_tokens]; sequence s owns
 *                [cu_seqlens[s], cu_seqlens[s + 1]).
 * cu_seqlens     device int32 [num_seqs + 1], ascending.
 * parent_hashes  device [num_seqs][32] bytes (16-byte aligned) continuing
 *                earlier chains, or NULL.
 * block_offsets  device int64 [num_seqs]: sequence s writes its k-th block
 *                hash to hashes[block_offsets[s] + k].
 * hashes         device [total_blocks][32] bytes (16-byte aligned), digests
 *                in the standard's big-endian byte order.
 * Device checks: bad cu_seqlens or a sequence whose hashes would pass
 * total_blocks -> PKV_DEVERR_CONTEXT, that sequence writes nothing.
 * One thread per sequence (the chain is sequential); one launch.
 * ------------------------------------------------------------------------- */
pkv_status pkv_block_hashes(const int32_t* token_ids, const int32_t* cu_seqlens,
                            int32_t num_seqs, int64_t total_tokens, int32_t block_size,
                            const uint8_t* parent_hashes, const int64_t* block_offsets,
                            int64_t total_blocks, uint8_t* hashes, int32_t* dev_err,
                            pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * Decode attention -- one query token per sequence attends over its whole
 * cached context, which the kernel reads block by block through the table.
 *   「KV 缓存与分页注意力」 §02 and §07; grouped heads: §11.
 *
 * For sequence s and query head h, with kv head g = h / (num_heads /
 * num_kv_heads) (consecutive query heads share a KV head) and c = context_lens[s]:
 *   k_t = K[block_tables[s][t / bs]][g][t % bs][:] * k_scale,  t in [0, c)
 *   v_t = V[...same...] * v_scale
 *   x_t = scale * dot(q[s][h], k_t)
 *   out[s][h][:] = sum_t exp(x_t - max x) v_t / sum_t exp(x_t - max x)
 * computed with fp32 accumulation and rounded once (to nearest even) to
 * q_dtype.  A context of length 0 gives out = 0.
 *
 * q             device [num_seqs][num_heads][head_dim] of q_dtype (F16/BF16).
 * block_tables  device int32 [num_seqs][max_blocks_per_seq]; entries past
 *               ceil(c / block_size) are never read.
 * context_lens  device int32 [num_seqs].
 * max_context_len  host upper bound of context_lens (sizes the grid and the
 *               workspace); a longer context is flagged and its output zeroed.
 * partition_size   tokens per split-context partition, a multiple of
 *               block_size, or 0 for the library's choice
 *               (pkv_decode_partition_size).  Contexts longer than one
 *               partition are processed as independent partitions whose
 *               partial results a log-sum-exp reduce merges.
 * workspace     device scratch of at least pkv_decode_workspace_bytes(...)
 *               bytes, 256-byte aligned; may be NULL when that size is 0.
 * out           device [num_seqs][num_heads][head_dim] of q_dtype.
 * Launches: one partition kernel, then (when max_context_len exceeds one
 *   partition) the reduce kernel, chained with programmatic dependent launch.
 *   The partition kernel of single-head (and FP8) items is itself launched
 *   that way, so that it overlaps the end of a kv_append before it; it reads
 *   nothing until the preceding kernel in the stream has finished.
 * Reproducibility: the same inputs and partition size give the same output
 *   bits on every call, whatever order the work items run in.
 * ------------------------------------------------------------------------- */
/* The partition size a decode of this shape uses: `requested` when positive,
 * else the library's choice.  With at most 128 sequences and contexts of at
 * most 8192 tokens, work items are num_seqs * num_heads when every query head
 * has its own KV head or the cache is FP8, num_seqs * num_kv_heads when a
 * 16-bit cache's KV heads serve groups of 2..16; with W = 3x the SM count:
 * items >= 2W -> one partition per context (no reduce); W <= items < 2W ->
 * one partition per context for the first kind, and 3/4 of max_context_len
 * (rounded up to the block size) for the grouped kind, so that only the
 * longest contexts are cut in two.  Otherwise about 256 KiB of K+V per KV head
 * and partition (1 MiB for the grouped case). */
int32_t pkv_decode_partition_size(const pkv_cache_desc* cache, int32_t num_seqs,
                                  int32_t num_heads, int32_t max_context_len,
                                  int32_t requested);

size_t pkv_decode_workspace_bytes(const pkv_cache_desc* cache, int32_t num_seqs,
                                  int32_t num_heads, int32_t max_context_len,
                                  int32_t partition_size);

pkv_status pkv_paged_attention_decode(const pkv_cache_desc* cache,
                                      const void* q, int32_t q_dtype,
                                      int32_t num_seqs, int32_t num_heads,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* context_lens, int32_t max_context_len,
                                      float scale, int32_t partition_size,
                                      void* workspace, size_t workspace_bytes,
                                      int32_t* dev_err, void* out, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * The two stages of pkv_paged_attention_decode, for callers (and timers) that
 * schedule them separately.  Arguments mean the same as above.
 *
 * Workspace layout (fp32, P = ceil(max_context_len / partition_size)):
 *   m[num_seqs][num_heads][P]   at byte 0
 *   l[num_seqs][num_heads][P]   at byte round_up(4*S*H*P, 256)
 *   o[num_seqs][num_heads][P][head_dim] at byte 2*round_up(4*S*H*P, 256)
 * For partition p (tokens [p*partition_size, (p+1)*partition_size) of c):
 *   m = max_t x_t * log2(e),  l = sum_t 2^(x_t*log2(e) - m),
 *   o = sum_t 2^(x_t*log2(e) - m) * v_t.
 * pkv_paged_attention_partitions writes these for every (s, h, p) of a
 * context longer than one partition, and writes out[s][h] directly for a
 * context of at most one partition.  pkv_lse_reduce merges, for every (s, h)
 * whose context spans two or more partitions,
 *   out = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p,  M = max_p m_p,
 * and leaves the other rows of out untouched.
 * ------------------------------------------------------------------------- */
pkv_status pkv_paged_attention_partitions(const pkv_cache_desc* cache,
                                          const void* q, int32_t q_dtype,
                                          int32_t num_seqs, int32_t num_heads,
                                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                                          const int32_t* context_lens, int32_t max_context_len,
                                          float scale, int32_t partition_size,
                                          void* workspace, size_t workspace_bytes,
                                          int32_t* dev_err, void* out, pkv_stream_t stream);

pkv_status pkv_lse_reduce(int32_t num_seqs, int32_t num_heads, int32_t head_dim,
                          const int32_t* context_lens, int32_t max_context_len,
                          int32_t partition_size, const void* workspace,
                          size_t workspace_bytes, int32_t out_dtype, void* out,
                          pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * Shared-prefix decode -- the decode above for a batch in which groups of
 * sequences share their leading blocks, as forked sequences do (parallel
 * sampling and beam search share the prompt's blocks by reference count:
 * 「KV 缓存与分页注意力」 §08 写时复制).  The result is the attention defined
 * above; only the reads change: a shared block is read once per group, KV head
 * and 8 or 16 query rows (members x query heads of the KV head) instead of
 * once per member and query head.
 *
 * Attention over [0, c) splits exactly at the end P of the shared prefix: the
 * prefix kernel writes (m, l, o) partials of [0, P) for every member and head,
 * the partition kernel those of [P, c), and the log-sum-exp reduce merges them.
 *
 * Groups: sequences [group_begin[i], group_begin[i + 1]) form group i.
 * group_begin          device int32 [num_groups + 1], ascending, starting at 0
 *                      and ending at num_seqs; every sequence is in one group
 *                      (a sequence that shares nothing is a group of one with
 *                      no prefix).
 * group_prefix_blocks  device int32 [num_groups]: P_i / block_size, the number
 *                      of leading block-table entries that every member of
 *                      group i holds equal to its first member's (0: nothing
 *                      shared).  Each member's context must hold at least
 *                      P_i tokens.
 * max_group_size, max_prefix_blocks  host upper bounds that size the prefix
 *                      kernel's grid, like max_context_len;
 *                      max_prefix_blocks * block_size <= max_context_len and
 *                      max_prefix_blocks <= max_blocks_per_seq.
 * workspace            at least pkv_shared_prefix_workspace_bytes(...) bytes
 *                      (the decode layout above with four more partials per
 *                      row: a shared prefix of P tokens is cut into at most
 *                      four partitions of round_up(ceil(max_prefix_blocks *
 *                      block_size / 4), block_size) tokens, which come before
 *                      the partitions of the rest of the context).
 * Device checks (with dev_err): a group entry out of range or a prefix above
 * max_prefix_blocks flags PKV_DEVERR_PREFIX and that group's prefix is not
 * computed (its members' outputs are then zero, flagged PKV_DEVERR_CONTEXT,
 * as far as the group's bounds can be used); a member past max_group_size or
 * with a context shorter than its prefix flags PKV_DEVERR_CONTEXT and its
 * output is zero; a member whose table differs from the first member's inside
 * the prefix flags PKV_DEVERR_PREFIX (its output then uses the first member's
 * blocks).
 * Supported: F16 or BF16 caches with q of the same type, 1..16 query heads per
 * KV head; anything else returns PKV_ERR_UNSUPPORTED and launches nothing.
 * num_groups == 0 or max_prefix_blocks == 0 gives the plain decode.
 * Launches: with partition_size 0, max_context_len <= 4096 and at least one
 *   (group, KV head, row tile) per SM, one kernel: each CTA reads its group's
 *   shared blocks once for its rows, then each member's own blocks for that
 *   member's rows, keeps one online softmax per row and writes out (the
 *   workspace is not touched).  Otherwise three: prefix kernel, partition
 *   kernel, reduce.  Both compute the attention defined above.
 * ------------------------------------------------------------------------- */
size_t pkv_shared_prefix_workspace_bytes(const pkv_cache_desc* cache, int32_t num_seqs,
                                         int32_t num_heads, int32_t max_context_len,
                                         int32_t partition_size);

pkv_status pkv_paged_attention_decode_shared_prefix(
    const pkv_cache_desc* cache, const void* q, int32_t q_dtype, int32_t num_seqs,
    int32_t num_heads, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* context_lens, int32_t max_context_len, int32_t num_groups,
    const int32_t* group_begin, const int32_t* group_prefix_blocks, int32_t max_group_size,
    int32_t max_prefix_blocks, float scale, int32_t partition_size, void* workspace,
    size_t workspace_bytes, int32_t* dev_err, void* out, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * Prefill attention -- the prompt phase: all new tokens of each sequence
 * attend causally over the paged cache (「KV Cache从原理到实战」 §2.3: the
 * prompt's K and V are computed and stored in one pass; 「KV 缓存与分页注意力」
 * §02: a token attends to itself and every earlier token).
 *
 * The new tokens' K/V must already be in the cache (pkv_kv_append), as the
 * last n_s of each context.  For sequence s, n_s = cu_seqlens_q[s + 1] -
 * cu_seqlens_q[s] and c = context_lens[s]; query row cu_seqlens_q[s] + j
 * (j < n_s) sits at position p = c - n_s + j and
 *   out[row][h][:] = sum_{t <= p} exp(x_t - max x) v_t / sum_{t <= p} exp(x_t - max x),
 *   x_t = scale * dot(q[row][h], k_t),  k_t, v_t of KV head h / (num_heads / num_kv_heads)
 * with fp32 accumulation, rounded once to q_dtype.  A context cached before
 * the new tokens (chunked prefill) is attended to like the rest.
 *
 * q, out        device [total_q][num_heads][head_dim] of q_dtype, 16-byte aligned.
 * cu_seqlens_q  device int32 [num_seqs + 1], ascending from 0 to total_q.
 * max_q_len     host upper bound of n_s (sizes the grid).
 * block_tables, context_lens, max_context_len: as for the decode.
 * Supported: F16 or BF16 caches with q of the same type, head_dim 64 or 128,
 *   block_size 8, 16 or 32, 1..128 query heads per KV head; others return
 *   PKV_ERR_UNSUPPORTED.
 * Device checks (with dev_err): n_s above max_q_len or c, c above
 *   max_context_len or the table, bad cu_seqlens_q -> PKV_DEVERR_CONTEXT (that
 *   sequence's rows are zero, or untouched when cu_seqlens_q is bad); a bad block
 *   id -> PKV_DEVERR_BLOCK_ID (the key is read as zeros).
 * Launches: one kernel.
 * ------------------------------------------------------------------------- */
pkv_status pkv_paged_attention_prefill(const pkv_cache_desc* cache, const void* q,
                                       int32_t q_dtype, int32_t num_seqs, int32_t num_heads,
                                       const int32_t* cu_seqlens_q, int32_t total_q,
                                       int32_t max_q_len, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* context_lens,
                                       int32_t max_context_len, float scale, int32_t* dev_err,
                                       void* out, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_paged_attention_decode_static_ws -- the decode above for callers that
 * cannot allocate device memory.  The pages have no counterpart: this is a
 * deployment convenience of the library, not part of the method.
 *
 * Some callers cannot call cudaMalloc or pass a workspace: an engine that has
 * reserved nearly all of the GPU's memory up front for its own KV-cache pool
 * (a cudaMalloc would then fail), or code on a latency-critical path where
 * cudaMalloc / cudaFree may synchronise the device.  This entry point takes
 * the split-context partials from a static device array of
 * PKV_STATIC_SCRATCH_BYTES inside the library and allocates nothing (no
 * cudaMalloc, no cudaFree, no allocating library routine).
 *
 * Arguments and results: those of pkv_paged_attention_decode, without the
 * workspace.  The caller still owns and passes q, the tables, dev_err, out.
 * - Limit: a request with pkv_decode_workspace_bytes(...) above
 *   PKV_STATIC_SCRATCH_BYTES returns PKV_ERR_SCRATCH_LIMIT and launches nothing.
 * - Every GPU that loads the library holds the array until the process exits.
 * - The first call on a device, with that device current, looks up the array's
 *   device address (cudaGetSymbolAddress) and caches it for later calls; make
 *   that first call before any stream capture.
 * - All calls share the one array, which keeps the last call's contents.
 *   Nothing in it needs to start at zero: each call writes every partial it
 *   reads.  Calls whose kernels can overlap on the GPU (different streams,
 *   different host threads) race on the array; issue them on one stream.
 * ------------------------------------------------------------------------- */
#define PKV_STATIC_SCRATCH_BYTES ((size_t)32 << 20)
/* (The address looked up on a device's first call belongs to that device's
 * CUDA context: after cudaDeviceReset, do not call this entry point again in
 * the same process.) */

pkv_status pkv_paged_attention_decode_static_ws(const pkv_cache_desc* cache,
                                                const void* q, int32_t q_dtype,
                                                int32_t num_seqs, int32_t num_heads,
                                                const int32_t* block_tables,
                                                int32_t max_blocks_per_seq,
                                                const int32_t* context_lens,
                                                int32_t max_context_len, float scale,
                                                int32_t partition_size, int32_t* dev_err,
                                                void* out, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_testing_set_decode_wait_limit -- a testing aid, not part of the method
 * (the pages have no counterpart).
 *
 * The streaming decode kernel waits on mbarriers for its own bulk copies, and
 * every such wait is bounded: after the limit it sets PKV_DEVERR_TIMEOUT in
 * dev_err, stops waiting everywhere, lets the copies it started land and
 * returns, so the context stays usable.  This call sets the number of polls
 * per wait for decode calls issued afterwards (captured into their launch
 * parameters at the call): 0 restores the kernel's own limit (2^22 polls, and
 * at most one second from a wait's first failed poll).  Under a lower limit a
 * poll is one look at the barrier that does not suspend the thread, so a wait
 * that is not already complete runs out.  A test sets a small value to make a
 * wait run out on purpose and check the error path.  Returns the previous
 * setting.  Process-wide; the drain of copies in flight always keeps the full
 * limit.
 * ------------------------------------------------------------------------- */
uint32_t pkv_testing_set_decode_wait_limit(uint32_t tries);

/* ---------------------------------------------------------------------------
 * pkv_testing_set_shared_prefix_path -- a testing aid, not part of the method
 * (the pages have no counterpart).
 *
 * pkv_paged_attention_decode_shared_prefix computes the same attention by one
 * of two routes: a single pass (one kernel; each CTA reads a group's shared
 * blocks once for its rows, then each member's own blocks, and writes out
 * directly), or a split (prefix kernel + partition kernel + log-sum-exp
 * reduce over the workspace).  The library takes the single pass when
 * partition_size is 0, max_context_len <= 4096 and the single pass has at
 * least one CTA per SM; the split otherwise.  This call overrides that choice
 * for later calls: 0 = the library's choice, 1 = always the single pass (the
 * partition size is then unused), 2 = always the split.  Returns the previous
 * setting, or -1 (and changes nothing) for another value.  Process-wide.
 * ------------------------------------------------------------------------- */
int32_t pkv_testing_set_shared_prefix_path(int32_t path);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
