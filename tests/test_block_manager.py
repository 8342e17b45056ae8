"""Host block bookkeeping: on-demand blocks, the waste bound, sharing and
copy-on-write, against the worked examples the pages print."""
import json
import os

import numpy as np
import pytest

from paged_kv_cache_130_gb300.block_manager import BlockManager, BlockPool, OutOfBlocks
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
