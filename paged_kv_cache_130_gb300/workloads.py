"""Seeded synthetic workloads for the decode path (inputs only).

Each workload is one decode layer: a pre-filled paged cache, the step's new
tokens with their slots, the query of every sequence, the block tables and the
context lengths after the step, and -- for parallel sampling -- the
copy-on-write block pairs.  Both the CUDA path and the CPU oracle take their
inputs from here; this module holds none of the attention arithmetic.

Values are drawn with numpy's PCG64 from a seed, in float32, and rounded to the
I/O type (fp16 through numpy, bf16 through torch's CPU cast, both round to
nearest even).  Every array of element data holds raw bits: uint16 for fp16 and
bf16.  Prefill values are drawn per segment (one sequence, or one shared prompt)
from their own sub-seed, so any one sequence can be rebuilt without the others.

Workload shapes (the five decode layers of the benchmark):

=========================  =========================================================
tiny_f16                   fp16, 8 heads = 8 KV heads, head_dim 64, block 16, 4
                           sequences of 5/17/33/64 tokens, pool 64 blocks
opt13b_f16                 OPT-13B layer: fp16, 40 x 128 MHA, block 16, batch 32,
                           log-normal lengths (median 500, sigma 0.5, clip
                           [1, 2048]), pool sized for 15,700 tokens (grown if the
                           draw needs more), values 0.5 N(0,1)
llama2_70b_bf16_gqa        Llama-2-70B layer: bf16, 64 query / 8 KV heads x 128,
                           block 16, batch 64, lengths U[1024, 4096]
cow_parallel_sampling_f16  fp16, 32 x 128, block 16, 16 prompts x 6 samples,
                           shared 504-token prompt (last block half full), tails
                           U[1, 256]; the step copies the shared last block for
                           five of the six samples, appends every tail, decodes
                           all 96 sequences
llama2_7b_fp8_long         Llama-2-7B layer: E4M3 cache with one fp32 scale per
                           tensor (K, V), bf16 q / inputs, 32 x 128, block 32,
                           batch 16, lengths U[8192, 32768], 512-token partitions
=========================  =========================================================

The sizes come from the pages: OPT-13B's 5,120-wide layer and the 12 GB /
15,700-token cache budget (「KV 缓存与分页注意力」 §03), Llama-2-70B's 64 query
heads over 8 KV heads (same page, §11), Llama-2-7B's 4,096 width
(「KV Cache从原理到实战」 §2.2), the 16-token default block (first page, §06),
parallel samples sharing prompt blocks with copy-on-write (first page, §08) and
8-bit float caches (first page, §11).
"""
from dataclasses import dataclass, field
import math

import numpy as np

from .block_manager import BlockManager, BlockPool, shared_prefix_groups

F16, BF16, E4M3 = 0, 1, 2
DTYPE_NAMES = {F16: "f16", BF16: "bf16", E4M3: "e4m3"}
E4M3_MAX = 448.0


def _rng(*key):
    return np.random.Generator(np.random.PCG64(list(key)))


def _to_bits(x32, code):
    """Round float32 values to fp16 / bf16 (nearest even) and return the bits."""
    if code == F16:
        return x32.astype(np.float16).view(np.uint16)
    if code == BF16:
        import torch
        t = torch.from_numpy(np.ascontiguousarray(x32)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    raise ValueError("inputs are fp16 or bf16")


def bits_to_float32(bits, code):
    """Exact float32 value of fp16 / bf16 bits (for scale calibration only)."""
    if code == F16:
        return bits.view(np.float16).astype(np.float32)
    if code == BF16:
        return (bits.astype(np.uint32) << 16).view(np.float32)
    raise ValueError(code)


@dataclass
class Segment:
    """A run of prefill tokens written with one draw of values."""
    key: tuple
    slots: np.ndarray          # int64 [n]


@dataclass
class Workload:
    name: str
    seed: int
    cache_dtype: int
    io_dtype: int
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    value_sigma: float
    scale: float                       # softmax scale, an fp32 value
    partition_size: int                # 0 = library default
    context_lens: np.ndarray           # int32 [S], after the step
    block_tables: np.ndarray           # int32 [S, max_blocks]
    q: np.ndarray                      # uint16 [S, H, D]
    segments: list                     # prefill segments
    step_slots: np.ndarray             # int64 [T]
    step_key: tuple
    copy_pairs: np.ndarray             # int64 [n, 2]
    k_scale: float = 1.0
    v_scale: float = 1.0
    notes: dict = field(default_factory=dict)
    # prefill workloads: int32 [S + 1]; q is then [total_q, H, D] and the step
    # appends every new token before the prefill attention
    cu_seqlens_q: np.ndarray = None

    # ------------------------------------------------------------ values
    def values(self, key, n):
        """(k, v) bits [n, Hkv, D] of the segment / step with this key."""
        shape = (n, self.num_kv_heads, self.head_dim)
        r = _rng(self.seed, *key)
        k = r.standard_normal(shape, dtype=np.float32) * np.float32(self.value_sigma)
        v = r.standard_normal(shape, dtype=np.float32) * np.float32(self.value_sigma)
        return _to_bits(k, self.io_dtype), _to_bits(v, self.io_dtype)

    def step_values(self):
        return self.values(self.step_key, len(self.step_slots))

    def prefill(self, threads=1, segments=None):
        """Iterate (slots, k_bits, v_bits) over the prefill segments (or the
        given ones), in order.  With threads > 1 the values of the next
        segments are drawn ahead in a thread pool (each segment has its own
        generator, so the values are the same either way)."""
        segs = self.segments if segments is None else segments
        if threads <= 1:
            for seg in segs:
                k, v = self.values(seg.key, len(seg.slots))
                yield seg.slots, k, v
            return
        import concurrent.futures as cf
        ahead = 2 * threads
        with cf.ThreadPoolExecutor(threads) as ex:
            futs = [ex.submit(self.values, sg.key, len(sg.slots)) for sg in segs[:ahead]]
            for i, seg in enumerate(segs):
                k, v = futs[i].result()
                futs[i] = None
                if i + ahead < len(segs):
                    nxt = segs[i + ahead]
                    futs.append(ex.submit(self.values, nxt.key, len(nxt.slots)))
                yield seg.slots, k, v

    def segment_sequences(self, seg):
        """Sequences whose context holds a prefill segment's tokens: one
        sequence, or every sample of a shared prompt."""
        tails = self.notes.get("tails")
        if tails is not None:
            samples = int(tails.shape[1])
            p = seg.key[1]
            return set(range(p * samples, (p + 1) * samples))
        return {seg.key[1]}

    def segments_of(self, seqs):
        """The prefill segments that the given sequences read."""
        want = set(int(s) for s in seqs)
        return [seg for seg in self.segments if self.segment_sequences(seg) & want]

    # ------------------------------------------------------------ sizes
    @property
    def max_blocks_per_seq(self):
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self):
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def cache_elem_bytes(self):
        return 1 if self.cache_dtype == E4M3 else 2

    @property
    def io_elem_bytes(self):
        return 2

    def kv_bytes(self):
        """K/V bytes one decode reads: every cached element once per KV head."""
        ctx = self.context_lens.astype(np.int64)
        return int(ctx.sum()) * self.num_kv_heads * self.head_dim * 2 * self.cache_elem_bytes

    def decode_bytes(self):
        """Algorithmic bytes of one decode call: every cached K/V element read
        once per KV head, q and out once, the used block-table entries and the
        context lengths."""
        ctx = self.context_lens.astype(np.int64)
        kv = int(ctx.sum()) * self.num_kv_heads * self.head_dim * 2 * self.cache_elem_bytes
        qo = 2 * self.num_seqs * self.num_heads * self.head_dim * self.io_elem_bytes
        bt = 4 * int(((ctx + self.block_size - 1) // self.block_size).sum())
        return kv + qo + bt + 4 * self.num_seqs

    def unique_kv_bytes(self):
        """K/V bytes of the distinct physical blocks the decode touches,
        counted at the tokens they hold (shared prompt blocks once)."""
        seen = {}
        for s in range(self.num_seqs):
            ctx = int(self.context_lens[s])
            nblk = (ctx + self.block_size - 1) // self.block_size
            for i in range(nblk):
                fill = min(self.block_size, ctx - i * self.block_size)
                b = int(self.block_tables[s, i])
                seen[b] = max(seen.get(b, 0), fill)
        tokens = sum(seen.values())
        return tokens * self.num_kv_heads * self.head_dim * 2 * self.cache_elem_bytes

    def prefix_groups(self):
        """(group_begin, prefix_blocks) of the batch's shared prefixes: runs of
        consecutive sequences whose block tables start with the same blocks."""
        return shared_prefix_groups(self.block_tables, self.context_lens, self.block_size)

    def prefill_flops(self):
        """Multiply-adds x 2 of the causal prefill: query j of sequence s at
        position p reads p + 1 keys and values, 2 (p + 1) D MACs per head."""
        cu = self.cu_seqlens_q.astype(np.int64)
        ctx = self.context_lens.astype(np.int64)
        total = 0
        for s in range(self.num_seqs):
            n = int(cu[s + 1] - cu[s])
            first = int(ctx[s]) - n + 1               # keys of the first new token
            total += n * first + n * (n - 1) // 2     # sum of keys over the n rows
        return 4 * total * self.head_dim * self.num_heads

    @property
    def max_q_len(self):
        return int(np.diff(self.cu_seqlens_q).max()) if self.num_seqs else 0

    @property
    def total_q(self):
        return int(self.cu_seqlens_q[-1])

    def append_bytes(self):
        t = int((self.step_slots >= 0).sum())
        per = self.num_kv_heads * self.head_dim * 2 * (self.io_elem_bytes + self.cache_elem_bytes)
        return t * (per + 8)

    def copy_bytes(self):
        blk = self.num_kv_heads * self.block_size * self.head_dim * self.cache_elem_bytes
        return int(self.copy_pairs.shape[0]) * 2 * 2 * blk

    # ------------------------------------------------------------ scales
    def calibrate_fp8_scales(self, threads=None):
        """One scale per tensor: amax of every value written / 448 (fp32).
        The segments are drawn in a thread pool (a maximum does not depend on
        the order)."""
        if self.cache_dtype != E4M3:
            return
        import concurrent.futures as cf
        import os

        def amax(key, n):
            k, v = self.values(key, n)
            return (np.abs(bits_to_float32(k, self.io_dtype)).max(initial=0),
                    np.abs(bits_to_float32(v, self.io_dtype)).max(initial=0))

        jobs = [(seg.key, len(seg.slots)) for seg in self.segments]
        jobs.append((self.step_key, len(self.step_slots)))
        if threads is None:
            threads = min(16, os.cpu_count() or 1)
        with cf.ThreadPoolExecutor(max(1, threads)) as ex:
            found = list(ex.map(lambda j: amax(*j), jobs))
        amax_k = np.float32(max((a for a, _ in found), default=0.0))
        amax_v = np.float32(max((b for _, b in found), default=0.0))
        self.k_scale = float(np.float32(amax_k) / np.float32(E4M3_MAX)) if amax_k > 0 else 1.0
        self.v_scale = float(np.float32(amax_v) / np.float32(E4M3_MAX)) if amax_v > 0 else 1.0


# ---------------------------------------------------------------- builders

def _pool_and_manager(num_blocks, block_size, seed):
    order = _rng(seed, 9).permutation(num_blocks)
    pool = BlockPool(num_blocks, block_size, order=order)
    return pool, BlockManager(pool)


def _independent(name, seed, cache_dtype, io_dtype, num_heads, num_kv_heads, head_dim,
                 block_size, ctx, value_sigma, num_blocks=None, pool_factor=1.25,
                 min_blocks=0, partition_size=0, max_seg_tokens=4096):
    """Sequences with independent contexts: prefill ctx-1 tokens, the step
    appends each sequence's last token, decode over ctx tokens."""
    ctx = np.asarray(ctx, dtype=np.int64)
    need = int(((ctx + block_size - 1) // block_size).sum())
    if num_blocks is None:
        num_blocks = max(min_blocks, int(math.ceil(pool_factor * need)))
    pool, mgr = _pool_and_manager(num_blocks, block_size, seed)
    seqs = [mgr.new_sequence() for _ in ctx]
    segments = []
    for i, (s, n) in enumerate(zip(seqs, ctx)):
        slots, pairs = mgr.append_tokens(s, int(n) - 1)
        assert not pairs
        for j in range(0, len(slots), max_seg_tokens):
            segments.append(Segment(key=(1, i, j // max_seg_tokens),
                                    slots=slots[j:j + max_seg_tokens]))
    step = np.empty(len(seqs), dtype=np.int64)
    for i, s in enumerate(seqs):
        step[i], pair = mgr.append_slot(s)
        assert pair is None
    tables = BlockManager.block_table_array(seqs)
    q = _to_bits(_rng(seed, 3).standard_normal((len(seqs), num_heads, head_dim),
                                                 dtype=np.float32) * np.float32(value_sigma),
                 io_dtype)
    w = Workload(name=name, seed=seed, cache_dtype=cache_dtype, io_dtype=io_dtype,
                 num_seqs=len(seqs), num_heads=num_heads, num_kv_heads=num_kv_heads,
                 head_dim=head_dim, block_size=block_size, num_blocks=num_blocks,
                 value_sigma=value_sigma,
                 scale=float(np.float32(1.0) / np.float32(math.sqrt(head_dim))),
                 partition_size=partition_size,
                 context_lens=ctx.astype(np.int32), block_tables=tables, q=q,
                 segments=segments, step_slots=step, step_key=(2,),
                 copy_pairs=np.zeros((0, 2), dtype=np.int64))
    w.notes["blocks_needed"] = need
    w.notes["pool_blocks"] = num_blocks
    w.notes["refcount_max"] = int(pool.refcount.max()) if num_blocks else 0
    return w


def tiny_f16(seed=1, ctx=(5, 17, 33, 64)):
    return _independent("tiny_f16", seed, F16, F16, 8, 8, 64, 16, ctx, 1.0,
                        num_blocks=64)


def opt13b_f16(seed=2, num_seqs=32, median=500.0, sigma=0.5, max_len=2048):
    z = _rng(seed, 0).standard_normal(num_seqs)
    ctx = np.clip(np.rint(np.exp(math.log(median) + sigma * z)), 1, max_len).astype(np.int64)
    # a 12 GB / 819,200-byte budget holds 15,700 tokens = 982 blocks of 16;
    # the pool grows to the draw's need when that is larger
    w = _independent("opt13b_f16", seed, F16, F16, 40, 40, 128, 16, ctx, 0.5,
                     pool_factor=1.0, min_blocks=int(math.ceil(15700 / 16)))
    w.notes["pool_rule"] = ("15,700-token budget" if w.num_blocks == 982
                            else "grown to the draw's block count")
    return w


def llama2_70b_bf16_gqa(seed=3, num_seqs=64, lo=1024, hi=4096):
    ctx = _rng(seed, 0).integers(lo, hi, size=num_seqs, endpoint=True)
    return _independent("llama2_70b_bf16_gqa", seed, BF16, BF16, 64, 8, 128, 16, ctx, 1.0)


def llama2_7b_fp8_long(seed=5, num_seqs=16, lo=8192, hi=32768, calibrate=True):
    ctx = _rng(seed, 0).integers(lo, hi, size=num_seqs, endpoint=True)
    w = _independent("llama2_7b_fp8_long", seed, E4M3, BF16, 32, 32, 128, 32, ctx, 1.0,
                     partition_size=512)
    if calibrate:
        w.calibrate_fp8_scales()
    return w


def cow_parallel_sampling_f16(seed=4, num_prompts=16, samples=6, prompt_len=504,
                              tail_lo=1, tail_hi=256, num_heads=32, head_dim=128,
                              block_size=16, num_kv_heads=None, dtype=F16,
                              name="cow_parallel_sampling_f16"):
    """Shared prompts with copy-on-write at the first divergent write.

    Set-up: each prompt's tokens are written once; ``samples`` sequences share
    its blocks (reference count ``samples``).  The step: every sample appends
    its tail; the first tail token of each of the first ``samples - 1`` samples
    finds the half-full last prompt block shared and gets a private copy (the
    (src, dst) pairs), the last sample writes in place.  ``copy_blocks`` runs
    before the append, the decode reads all sequences."""
    tails = _rng(seed, 0).integers(tail_lo, tail_hi, size=(num_prompts, samples),
                                   endpoint=True)

    def simulate(num_blocks, order_seed):
        if order_seed is None:
            pool = BlockPool(num_blocks, block_size)
            mgr = BlockManager(pool)
        else:
            pool, mgr = _pool_and_manager(num_blocks, block_size, order_seed)
        segs, seqs, step, pairs = [], [], [], []
        for p in range(num_prompts):
            root = mgr.new_sequence()
            slots, pp = mgr.append_tokens(root, prompt_len)
            assert not pp
            segs.append(Segment(key=(1, p, 0), slots=slots))
            group = [root] + [mgr.fork(root) for _ in range(samples - 1)]
            seqs.extend(group)
        refmax = int(pool.refcount.max())
        for i, s in enumerate(seqs):
            slots, pp = mgr.append_tokens(s, int(tails.reshape(-1)[i]))
            step.append(slots)
            pairs.extend(pp)
        used = num_blocks - pool.num_free
        return segs, seqs, np.concatenate(step), pairs, used, refmax, pool

    _, _, _, _, used, _, _ = simulate(10 ** 7, None)
    num_blocks = int(math.ceil(1.25 * used))
    segs, seqs, step, pairs, used, refmax, pool = simulate(num_blocks, seed)
    ctx = np.array([s.num_tokens for s in seqs], dtype=np.int64)
    tables = BlockManager.block_table_array(seqs)
    q = _to_bits(_rng(seed, 3).standard_normal((len(seqs), num_heads, head_dim),
                                                 dtype=np.float32), dtype)
    hkv = num_heads if num_kv_heads is None else num_kv_heads
    w = Workload(name=name, seed=seed, cache_dtype=dtype, io_dtype=dtype,
                 num_seqs=len(seqs), num_heads=num_heads, num_kv_heads=hkv,
                 head_dim=head_dim, block_size=block_size, num_blocks=num_blocks,
                 value_sigma=1.0,
                 scale=float(np.float32(1.0) / np.float32(math.sqrt(head_dim))),
                 partition_size=0, context_lens=ctx.astype(np.int32), block_tables=tables,
                 q=q, segments=segs, step_slots=step, step_key=(2,),
                 copy_pairs=np.array(pairs, dtype=np.int64).reshape(-1, 2))
    w.notes.update(blocks_used=used, pool_blocks=num_blocks, refcount_after_fork=refmax,
                   refcount_after_step=pool.refcount.copy(), tails=tails)
    return w


def _prompts(name, seed, dtype, num_heads, num_kv_heads, head_dim, block_size, new, cached,
             max_seg_tokens=4096):
    """Prompt-phase batches: sequence i holds cached[i] tokens from earlier
    chunks (written in the set-up), the step appends its new[i] tokens, then
    the prefill attention runs for the new tokens."""
    new = np.asarray(new, dtype=np.int64)
    cached = np.asarray(cached, dtype=np.int64)
    ctx = new + cached
    need = int(((ctx + block_size - 1) // block_size).sum())
    num_blocks = int(math.ceil(1.25 * need))
    pool, mgr = _pool_and_manager(num_blocks, block_size, seed)
    seqs = [mgr.new_sequence() for _ in ctx]
    segments, step = [], []
    for i, s in enumerate(seqs):
        slots, _ = mgr.append_tokens(s, int(cached[i]))
        for j in range(0, len(slots), max_seg_tokens):
            segments.append(Segment(key=(1, i, j // max_seg_tokens),
                                    slots=slots[j:j + max_seg_tokens]))
    for s, n in zip(seqs, new):
        slots, _ = mgr.append_tokens(s, int(n))
        step.append(slots)
    tables = BlockManager.block_table_array(seqs)
    cu = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    q = _to_bits(_rng(seed, 3).standard_normal((int(cu[-1]), num_heads, head_dim),
                                                 dtype=np.float32), dtype)
    w = Workload(name=name, seed=seed, cache_dtype=dtype, io_dtype=dtype,
                 num_seqs=len(seqs), num_heads=num_heads, num_kv_heads=num_kv_heads,
                 head_dim=head_dim, block_size=block_size, num_blocks=num_blocks,
                 value_sigma=1.0,
                 scale=float(np.float32(1.0) / np.float32(math.sqrt(head_dim))),
                 partition_size=0, context_lens=ctx.astype(np.int32), block_tables=tables,
                 q=q, segments=segments, step_slots=np.concatenate(step), step_key=(2,),
                 copy_pairs=np.zeros((0, 2), dtype=np.int64), cu_seqlens_q=cu)
    w.notes["pool_blocks"] = num_blocks
    return w


def prefill_llama2_7b_bf16(seed=6, num_seqs=8, lo=512, hi=2048, num_heads=32,
                           num_kv_heads=32, head_dim=128, block_size=16, dtype=BF16):
    """Llama-2-7B attention layer shape, whole prompts of U[lo, hi] tokens."""
    new = _rng(seed, 0).integers(lo, hi, size=num_seqs, endpoint=True)
    return _prompts("prefill_llama2_7b_bf16", seed, dtype, num_heads, num_kv_heads, head_dim,
                    block_size, new, np.zeros(num_seqs, np.int64))


def prefill_llama2_70b_gqa_chunked_bf16(seed=7, num_seqs=4, chunk=512, lo=1024, hi=4096,
                                        block_size=16):
    """Llama-2-70B layer shape (64 query heads over 8 KV heads), chunked
    prefill: U[lo, hi] tokens already cached, then a chunk of new tokens."""
    cached = _rng(seed, 0).integers(lo, hi, size=num_seqs, endpoint=True)
    return _prompts("prefill_llama2_70b_gqa_chunked_bf16", seed, BF16, 64, 8, 128, block_size,
                    np.full(num_seqs, chunk, np.int64), cached)


PREFILL_WORKLOADS = {
    "prefill_llama2_7b_bf16": prefill_llama2_7b_bf16,
    "prefill_llama2_70b_gqa_chunked_bf16": prefill_llama2_70b_gqa_chunked_bf16,
}


@dataclass
class SwapWorkload:
    """Pre-emption by swapping: the blocks of the `swapped` sequences of a
    decode batch leave the device pool for pinned host memory, every layer,
    and come back into free device blocks (「KV 缓存与分页注意力」 §09)."""
    name: str
    num_layers: int
    num_blocks: int             # device pool per layer
    host_blocks: int            # host pool per layer
    num_kv_heads: int
    block_size: int
    head_dim: int
    cache_dtype: int
    out_pairs: np.ndarray       # int64 [n, 2]: device block -> host block
    in_pairs: np.ndarray        # int64 [n, 2]: host block -> device block
    swapped_seqs: np.ndarray
    cu_seqlens_q: np.ndarray = None

    @property
    def block_bytes(self):
        return self.num_kv_heads * self.block_size * self.head_dim * (1 if self.cache_dtype == E4M3
                                                                       else 2)

    def swap_bytes(self):
        """Bytes one swap-out plus one swap-in move (each byte counted once):
        K and V of every pair and layer, both directions."""
        n = len(self.out_pairs) + len(self.in_pairs)
        return 2 * n * self.num_layers * self.block_bytes


def swap_opt13b_f16(seed=2, swapped=8, num_layers=40):
    """The OPT-13B decode batch (40 layers): its `swapped` longest sequences are
    swapped out and back in to the pool's free blocks."""
    w = opt13b_f16(seed=seed)
    order = np.argsort(-w.context_lens, kind="stable")[:swapped]
    blocks = []
    for s in order:
        n = (int(w.context_lens[s]) + w.block_size - 1) // w.block_size
        blocks.extend(int(b) for b in w.block_tables[s, :n])
    blocks = np.array(blocks, np.int64)
    used = set(int(b) for row, c in zip(w.block_tables, w.context_lens)
               for b in row[:(int(c) + w.block_size - 1) // w.block_size])
    free = np.array([b for b in range(w.num_blocks) if b not in used], np.int64)
    extra = len(blocks) - len(free)
    num_blocks = w.num_blocks + max(0, extra)
    if extra > 0:
        free = np.concatenate([free, np.arange(w.num_blocks, num_blocks)])
    host = np.arange(len(blocks), dtype=np.int64)
    dest = _rng(seed, 11).permutation(free)[:len(blocks)]
    return SwapWorkload(name="swap_opt13b_f16", num_layers=num_layers, num_blocks=num_blocks,
                        host_blocks=len(blocks), num_kv_heads=w.num_kv_heads,
                        block_size=w.block_size, head_dim=w.head_dim, cache_dtype=F16,
                        out_pairs=np.stack([blocks, host], 1),
                        in_pairs=np.stack([host, dest], 1), swapped_seqs=order)


SWAP_WORKLOADS = {"swap_opt13b_f16": swap_opt13b_f16}


@dataclass
class HashWorkload:
    """Prefix-cache hashing of a batch of prompts: the chained hash of every
    full block of token ids (「KV 缓存与分页注意力」 §11)."""
    name: str
    block_size: int
    token_ids: np.ndarray       # int32 [total_tokens]
    cu_seqlens: np.ndarray      # int32 [num_seqs + 1]
    cu_seqlens_q: np.ndarray = None

    @property
    def num_seqs(self):
        return len(self.cu_seqlens) - 1

    def full_blocks(self):
        return int((np.diff(self.cu_seqlens.astype(np.int64)) // self.block_size).sum())

    def hashed_token_bytes(self):
        """Token bytes that enter a hash (full blocks only)."""
        return 4 * self.block_size * self.full_blocks()


def hash_prompts(seed=8, num_seqs=4096, lo=512, hi=2048, block_size=16, vocab=32000):
    """4096 prompts of U[lo, hi] token ids drawn from a 32,000-entry vocabulary."""
    r = _rng(seed, 0)
    lens = r.integers(lo, hi, size=num_seqs, endpoint=True)
    toks = _rng(seed, 1).integers(0, vocab, size=int(lens.sum())).astype(np.int32)
    return HashWorkload(name="hash_prompts", block_size=block_size, token_ids=toks,
                        cu_seqlens=np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))


HASH_WORKLOADS = {"hash_prompts": hash_prompts}


WORKLOADS = {
    "tiny_f16": tiny_f16,
    "opt13b_f16": opt13b_f16,
    "llama2_70b_bf16_gqa": llama2_70b_bf16_gqa,
    "cow_parallel_sampling_f16": cow_parallel_sampling_f16,
    "llama2_7b_fp8_long": llama2_7b_fp8_long,
}


def make(name, **kw):
    if name in HASH_WORKLOADS:
        return HASH_WORKLOADS[name](**kw)
    if name in SWAP_WORKLOADS:
        return SWAP_WORKLOADS[name](**kw)
    if name in PREFILL_WORKLOADS:
        return PREFILL_WORKLOADS[name](**kw)
    return WORKLOADS[name](**kw)
