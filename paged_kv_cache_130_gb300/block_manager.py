"""Host-side block bookkeeping: pool, block tables, reference counts, copy-on-write.

This is the allocator that hands out the inputs of the device calls: the slot each
new token is written to (``slot_mapping``), the per-sequence block tables, and the
(src, dst) block pairs that ``copy_blocks`` must copy before a shared block is
written.  It does no attention arithmetic and never touches device memory.

Behaviour follows the pages:

* the cache is a pool of equal-size physical blocks; a sequence sees its blocks
  as logically contiguous while they sit anywhere in the pool
  (「KV 缓存与分页注意力」 §06 像内存分页);
* a block-table row maps logical block i to a physical block id; the fill count
  of each entry is not stored, it follows from the token count
  (same page, §07 块表);
* a new physical block is taken only when the previous one is full, so a
  sequence wastes fewer than ``block_size`` slots (same page, §07;
  「Paged Attention in LLMs」 worked example with block size 4);
* parallel samples share the prompt's blocks and each block counts its users;
  a sample about to write into a shared block first gets a private copy and the
  original's count drops by one (「KV 缓存与分页注意力」 §08 共用，写时复制);
* a finished sequence returns its blocks to the pool (same page, §07);
  running out of blocks raises, as the toy pager in
  「KV Cache从原理到实战」 §6.2 does.
"""
from collections import deque

import numpy as np


class OutOfBlocks(RuntimeError):
    """The pool has no free physical block left."""


class BlockPool:
    """Fixed pool of ``num_blocks`` physical blocks with reference counts.

    ``order`` fixes the order in which free blocks are handed out (a seeded
    permutation scatters a sequence's blocks over the pool)."""

    def __init__(self, num_blocks, block_size, order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        if order is None:
            order = range(self.num_blocks)
        order = [int(b) for b in order]
        if sorted(order) != list(range(self.num_blocks)):
            raise ValueError("order must be a permutation of the pool")
        self._free = deque(order)
        self.refcount = np.zeros(self.num_blocks, dtype=np.int64)

    @property
    def num_free(self):
        return len(self._free)

    def take(self):
        if not self._free:
            raise OutOfBlocks("out of KV cache blocks")
        b = self._free.popleft()
        self.refcount[b] = 1
        return b

    def share(self, b):
        if self.refcount[b] <= 0:
            raise ValueError("sharing a free block")
        self.refcount[b] += 1

    def release(self, b):
        if self.refcount[b] <= 0:
            raise ValueError("releasing a free block")
        self.refcount[b] -= 1
        if self.refcount[b] == 0:
            self._free.append(b)


class Sequence:
    """One sequence: its block table (physical ids, logical order) and length."""

    __slots__ = ("table", "num_tokens")

    def __init__(self, table=None, num_tokens=0):
        self.table = list(table or [])
        self.num_tokens = int(num_tokens)


class BlockManager:
    """Per-sequence block tables over one :class:`BlockPool`."""

    def __init__(self, pool):
        self.pool = pool

    @property
    def block_size(self):
        return self.pool.block_size

    def new_sequence(self):
        return Sequence()

    def append_slot(self, seq):
        """Reserve the slot of ``seq``'s next token.

        Returns ``(slot, pair)``: ``slot = block * block_size + offset`` and
        ``pair`` is ``(src, dst)`` when the write needs a copy-on-write of a
        shared block first, else ``None``."""
        bs = self.pool.block_size
        off = seq.num_tokens % bs
        pair = None
        if off == 0:
            # the last block is full (or there is none): take a fresh one
            seq.table.append(self.pool.take())
        else:
            last = seq.table[-1]
            if self.pool.refcount[last] > 1:
                fresh = self.pool.take()
                self.pool.release(last)
                seq.table[-1] = fresh
                pair = (last, fresh)
        slot = seq.table[-1] * bs + off
        seq.num_tokens += 1
        return slot, pair

    def append_tokens(self, seq, n):
        """Slots for ``n`` more tokens, and the copy pairs they trigger."""
        slots = np.empty(n, dtype=np.int64)
        pairs = []
        for i in range(n):
            slots[i], pair = self.append_slot(seq)
            if pair is not None:
                pairs.append(pair)
        return slots, pairs

    def fork(self, seq):
        """A new sequence that shares every block of ``seq`` (parallel sample)."""
        for b in seq.table:
            self.pool.share(b)
        return Sequence(seq.table, seq.num_tokens)

    def free(self, seq):
        for b in seq.table:
            self.pool.release(b)
        seq.table = []
        seq.num_tokens = 0

    @staticmethod
    def wasted_slots(seq, block_size):
        """Slots held by ``seq`` that hold no token (all in its last block)."""
        return len(seq.table) * block_size - seq.num_tokens

    @staticmethod
    def block_table_array(seqs, max_blocks=None, pad=-1):
        """int32 [num_seqs, max_blocks] table; entries past a sequence's last
        block are ``pad`` and are never read by the kernels."""
        mb = max((len(s.table) for s in seqs), default=0) if max_blocks is None else max_blocks
        out = np.full((len(seqs), max(mb, 1)), pad, dtype=np.int32)
        for i, s in enumerate(seqs):
            if len(s.table) > mb:
                raise ValueError("sequence holds more blocks than max_blocks")
            out[i, :len(s.table)] = s.table
        return out


def shared_prefix_groups(block_tables, context_lens, block_size):
    """Groups of consecutive sequences that share their leading blocks.

    Forked sequences hold the same physical blocks for the prompt they share
    (「KV 缓存与分页注意力」 §08 共用，写时复制): their block-table rows start
    with equal entries.  A group extends over the following rows while their
    first entry equals the group's first row's; its prefix is the number of
    leading entries every member holds equal to the first row's, counting only
    blocks that are full in every member (so that prefix * block_size tokens
    lie inside each member's context).

    Returns ``(group_begin, prefix_blocks)``: int32 arrays of ``num_groups + 1``
    and ``num_groups`` entries; rows [group_begin[i], group_begin[i + 1]) form
    group i.  A row that shares nothing is a group of one with prefix 0.
    """
    tables = np.asarray(block_tables)
    ctx = np.asarray(context_lens, dtype=np.int64)
    n = len(ctx)
    begin, prefix = [0], []
    i = 0
    while i < n:
        common = int(ctx[i] // block_size)
        j = i + 1
        while j < n and common > 0:
            full = int(ctx[j] // block_size)
            k = 0
            lim = min(common, full)
            while k < lim and tables[j, k] == tables[i, k]:
                k += 1
            if k == 0:
                break
            common = k
            j += 1
        prefix.append(common if j - i >= 2 else 0)
        begin.append(j)
        i = j
    return np.array(begin, dtype=np.int32), np.array(prefix, dtype=np.int32)
