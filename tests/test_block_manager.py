"""Host block bookkeeping: on-demand blocks, the waste bound, sharing and
copy-on-write, against the worked examples the pages print."""
import json
import os

import numpy as np
import pytest

from paged_kv_cache_130_gb300.block_manager import (BlockManager, BlockPool, OutOfBlocks,
                                                     shared_prefix_groups)
from paged_kv_cache_130_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_ten_token_reply_in_blocks_of_four():
    ex = _golden("paging_examples.json")["block_size_4_reply"]
    pool = BlockPool(16, ex["block_size"], order=[5, 12, 3] + [b for b in range(16)
                                                               if b not in (5, 12, 3)])
    mgr = BlockManager(pool)
    seq = mgr.new_sequence()
    slots, pairs = mgr.append_tokens(seq, ex["num_tokens"])
    assert seq.table == ex["block_table"] and not pairs
    assert len(seq.table) == ex["blocks"]
    assert BlockManager.wasted_slots(seq, ex["block_size"]) == ex["wasted_paged"]
    # slot of token t = table[t // 4] * 4 + t % 4
    assert list(slots) == [ex["block_table"][t // 4] * 4 + t % 4 for t in range(10)]


def test_new_block_only_when_previous_is_full():
    pool = BlockPool(64, 8, order=np.random.default_rng(1).permutation(64))
    mgr = BlockManager(pool)
    seq = mgr.new_sequence()
    for t in range(100):
        before = len(seq.table)
        mgr.append_slot(seq)
        assert len(seq.table) == before + (1 if t % 8 == 0 else 0)
        assert 0 <= BlockManager.wasted_slots(seq, 8) < 8


def test_two_answers_copy_on_write():
    ex = _golden("paging_examples.json")["cow_two_answers"]
    pool = BlockPool(8, ex["block_size"])
    mgr = BlockManager(pool)
    a = mgr.new_sequence()
    mgr.append_tokens(a, ex["prompt_tokens"])
    b = mgr.fork(a)
    assert len(a.table) == ex["shared_blocks"]
    assert all(pool.refcount[x] == ex["refcount_before"] for x in a.table)
    last = a.table[-1]
    slot, pair = mgr.append_slot(a)                 # first writer copies
    assert pair == (last, a.table[-1]) and a.table[-1] != last
    assert slot == a.table[-1] * ex["block_size"] + ex["prompt_tokens"] % ex["block_size"]
    assert pool.refcount[last] == ex["refcount_after_first_write"]
    slot, pair = mgr.append_slot(b)                 # now sole owner: writes in place
    assert pair is None and b.table[-1] == last
    assert a.table[0] == b.table[0] and pool.refcount[a.table[0]] == 2


def test_full_shared_block_needs_no_copy():
    pool = BlockPool(8, 4)
    mgr = BlockManager(pool)
    a = mgr.new_sequence()
    mgr.append_tokens(a, 8)                         # exactly two full blocks
    b = mgr.fork(a)
    _, pair = mgr.append_slot(a)
    assert pair is None and len(a.table) == 3 and len(b.table) == 2


def test_free_returns_blocks_and_exhaustion_raises():
    pool = BlockPool(3, 4)
    mgr = BlockManager(pool)
    a = mgr.new_sequence()
    mgr.append_tokens(a, 12)
    with pytest.raises(OutOfBlocks):
        mgr.append_slot(a)
    b = mgr.fork(a)
    mgr.free(a)
    assert pool.num_free == 0
    mgr.free(b)
    assert pool.num_free == 3 and pool.refcount.sum() == 0


def test_cow_workload_counts():
    w = W.cow_parallel_sampling_f16()
    assert w.num_seqs == 96
    assert w.notes["refcount_after_fork"] == 6
    assert w.copy_pairs.shape == (80, 2)            # 5 copies per prompt
    assert len(np.unique(w.copy_pairs[:, 1])) == 80
    assert not set(w.copy_pairs[:, 1]) & set(w.copy_pairs[:, 0])
    assert len(np.unique(w.copy_pairs[:, 0])) == 16
    # after the step every shared prompt block except the last is still held by 6
    rc = w.notes["refcount_after_step"]
    for p in range(16):
        table = w.block_tables[p * 6]
        assert all(rc[b] == 6 for b in table[:31])
    for s in range(96):
        assert 0 <= -(-int(w.context_lens[s]) // 16) * 16 - int(w.context_lens[s]) < 16


def test_cow_literal_512_prompt_copies_nothing():
    w = W.cow_parallel_sampling_f16(prompt_len=512, num_prompts=2)
    assert w.copy_pairs.shape == (0, 2)


def _check_groups(tables, ctx, bs, begin, prefix):
    """Every group's prefix is shared, full in every member, and maximal."""
    assert begin[0] == 0 and begin[-1] == len(ctx)
    assert np.all(np.diff(begin) >= 1) and len(prefix) == len(begin) - 1
    for i in range(len(prefix)):
        a, b, p = begin[i], begin[i + 1], int(prefix[i])
        if b - a == 1:
            assert p == 0
            continue
        for m in range(a, b):
            assert np.array_equal(tables[m, :p], tables[a, :p])
            assert p * bs <= ctx[m]
        # one more block would break sharing or leave some member's context
        grows = all(p + 1 <= ctx[m] // bs and tables[m, p] == tables[a, p] for m in range(a, b))
        assert not grows


def test_shared_prefix_groups_of_forked_prompts():
    w = W.cow_parallel_sampling_f16()
    begin, prefix = w.prefix_groups()
    assert np.array_equal(begin, np.arange(0, 97, 6))
    # 504-token prompts: 31 full shared blocks; the half-full 32nd was copied
    # by five of the six samples
    assert np.all(prefix == 31)
    _check_groups(w.block_tables, w.context_lens, 16, begin, prefix)


def test_shared_prefix_groups_without_forks_are_singletons():
    w = W.opt13b_f16(num_seqs=8)
    begin, prefix = w.prefix_groups()
    assert np.array_equal(begin, np.arange(9)) and np.all(prefix == 0)


def test_shared_prefix_groups_by_hand():
    bs = 4
    pool = BlockPool(64, bs)
    mgr = BlockManager(pool)
    a = mgr.new_sequence()
    mgr.append_tokens(a, 10)                # blocks 0, 1 full, block 2 half
    forks = [mgr.fork(a) for _ in range(2)]
    lone = mgr.new_sequence()
    mgr.append_tokens(lone, 9)
    c = mgr.new_sequence()
    mgr.append_tokens(c, 8)                 # exactly two full blocks
    d = mgr.fork(c)
    mgr.append_tokens(a, 3)                 # writes into the shared half block: copies
    mgr.append_tokens(forks[0], 1)
    mgr.append_tokens(d, 5)
    seqs = [a] + forks + [lone, c, d]
    tables = BlockManager.block_table_array(seqs)
    ctx = np.array([s.num_tokens for s in seqs])
    begin, prefix = shared_prefix_groups(tables, ctx, bs)
    assert begin.tolist() == [0, 3, 4, 6]
    # a's group shares 2 full blocks (the third was half full and is now
    # copied by a and by forks[0]); c and d share c's 2 blocks
    assert prefix.tolist() == [2, 0, 2]
    _check_groups(tables, ctx, bs, begin, prefix)


def test_shared_prefix_groups_random_forest():
    rng = np.random.default_rng(5)
    bs = 8
    pool = BlockPool(4096, bs, order=rng.permutation(4096))
    mgr = BlockManager(pool)
    seqs = []
    for _ in range(20):
        root = mgr.new_sequence()
        mgr.append_tokens(root, int(rng.integers(1, 60)))
        group = [root] + [mgr.fork(root) for _ in range(int(rng.integers(0, 4)))]
        for s in group:
            mgr.append_tokens(s, int(rng.integers(0, 20)))
        seqs.extend(group)
    tables = BlockManager.block_table_array(seqs)
    ctx = np.array([s.num_tokens for s in seqs])
    begin, prefix = shared_prefix_groups(tables, ctx, bs)
    _check_groups(tables, ctx, bs, begin, prefix)
