"""The seeded workload generator: shapes, determinism and invariants."""
import numpy as np
import pytest

from paged_kv_cache_130_gb300 import workloads as W


def _check_tables(w):
    bs = w.block_size
    seen = {}
    for s in range(w.num_seqs):
        ctx = int(w.context_lens[s])
        nblk = -(-ctx // bs)
        row = w.block_tables[s]
        assert np.all((row[:nblk] >= 0) & (row[:nblk] < w.num_blocks))
        assert np.all(row[nblk:] == -1)
        assert 0 <= nblk * bs - ctx < bs                 # waste < one block
        for i, b in enumerate(row[:nblk]):
            seen.setdefault(int(b), set()).add(s)
    return seen


def _all_slots(w):
    return np.concatenate([seg.slots for seg in w.segments] + [w.step_slots])


@pytest.mark.parametrize("name", ["tiny_f16", "opt13b_f16", "llama2_70b_bf16_gqa"])
def test_independent_sequences(name):
    w = W.make(name)
    seen = _check_tables(w)
    assert all(len(v) == 1 for v in seen.values())        # nothing shared
    slots = _all_slots(w)
    assert len(np.unique(slots)) == len(slots) == int(w.context_lens.sum())
    assert len(w.step_slots) == w.num_seqs
    # the step writes each sequence's last token
    for s in range(w.num_seqs):
        t = int(w.context_lens[s]) - 1
        assert w.step_slots[s] == w.block_tables[s, t // w.block_size] * w.block_size \
            + t % w.block_size


def test_tiny_shapes():
    w = W.tiny_f16()
    assert list(w.context_lens) == [5, 17, 33, 64]
    assert w.num_blocks == 64 and w.notes["blocks_needed"] == 10
    assert w.q.shape == (4, 8, 64) and w.q.dtype == np.uint16
    assert np.float32(w.scale) == np.float32(0.125)


def test_opt13b_pool_rule_and_lengths():
    w = W.opt13b_f16()
    assert w.num_blocks >= 982
    assert w.context_lens.min() >= 1 and w.context_lens.max() <= 2048
    assert w.num_blocks == max(982, w.notes["blocks_needed"])


def test_fp8_workload_scales_and_shapes():
    w = W.llama2_7b_fp8_long(num_seqs=2, lo=40, hi=90)
    assert w.cache_dtype == W.E4M3 and w.io_dtype == W.BF16 and w.block_size == 32
    assert w.partition_size == 512
    amax_k = max(np.abs(W.bits_to_float32(k, W.BF16)).max() for _, k, _ in w.prefill())
    amax_k = max(amax_k, np.abs(W.bits_to_float32(w.step_values()[0], W.BF16)).max())
    assert np.float32(w.k_scale) == np.float32(amax_k) / np.float32(448)


def test_values_are_deterministic_per_segment():
    a = W.tiny_f16()
    b = W.tiny_f16()
    for (sa, ka, va), (sb, kb, vb) in zip(a.prefill(), b.prefill()):
        assert np.array_equal(sa, sb) and np.array_equal(ka, kb) and np.array_equal(va, vb)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.block_tables, b.block_tables)


def test_byte_counts():
    w = W.tiny_f16()
    kv = (5 + 17 + 33 + 64) * 8 * 64 * 2 * 2
    assert w.decode_bytes() == kv + 2 * 4 * 8 * 64 * 2 + 4 * 10 + 16
    assert w.unique_kv_bytes() == kv
    c = W.cow_parallel_sampling_f16(num_prompts=2)
    assert c.unique_kv_bytes() < c.decode_bytes()
