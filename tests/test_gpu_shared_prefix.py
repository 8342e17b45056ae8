"""Shared-prefix decode against the oracle.

Forked sequences (parallel samples of one prompt) hold the prompt's physical
blocks by reference (「KV 缓存与分页注意力」 §08 共用，写时复制).  The shared-prefix
entry point reads those blocks once per group and splits each context at the
end of the shared prefix; the attention it returns is the same exact
attention, so the oracle's plain decode is the reference:
|gpu - oracle| <= 2e-3 + 2e-3 |oracle| (plus half a bf16 ulp for bf16 outputs).

The entry point has two routes, and every case runs through both: the single
pass (one kernel reads a group's shared blocks once for all its rows, then
each member's own blocks, and writes out) and the split (prefix kernel,
partition kernel over the rest of each context, log-sum-exp reduce).
"""
import numpy as np
import pytest
import torch

import harness as H
from paged_kv_cache_130_gb300 import binding as B
from paged_kv_cache_130_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    H.build_library()
    yield
    B.pkv_testing_set_shared_prefix_path(0)


PATHS = {"single_pass": 1, "split": 2}


@pytest.fixture(params=list(PATHS))
def route(request):
    """The shared-prefix route the test's calls take."""
    prev = B.pkv_testing_set_shared_prefix_path(PATHS[request.param])
    yield request.param
    B.pkv_testing_set_shared_prefix_path(prev)


def forked(**kw):
    base = dict(num_prompts=2, samples=6, prompt_len=504, tail_lo=1, tail_hi=256)
    base.update(kw)
    return W.cow_parallel_sampling_f16(**base)


def prepared(w):
    g = H.GpuRun(w)
    o = H.OracleRun(w)
    for r in (g, o):
        r.prefill()
        r.copy()
        r.step()
    torch.cuda.synchronize()
    assert np.array_equal(H.to_bits(g.k_cache), o.k_cache)
    return g, o


CASES = {
    # (workload kwargs, partition size)
    "mha_f16_one_pass": (dict(), 0),
    "mha_f16_small_partitions": (dict(), 64),
    "gqa8_bf16": (dict(num_heads=16, num_kv_heads=2, dtype=W.BF16), 0),
    "gqa8_bf16_small_partitions": (dict(num_heads=16, num_kv_heads=2, dtype=W.BF16), 128),
    "gqa16_bf16_three_samples": (dict(num_heads=32, num_kv_heads=2, dtype=W.BF16, samples=3),
                                 0),
    "gqa4_f16_d64_bs32": (dict(num_heads=16, num_kv_heads=4, head_dim=64, block_size=32,
                               prompt_len=500), 0),
    "mha_bf16_short_prompt": (dict(num_heads=8, dtype=W.BF16, prompt_len=40, tail_hi=20), 32),
}


@pytest.mark.parametrize("case", list(CASES))
def test_shared_prefix_matches_oracle(case, route):
    kw, ps = CASES[case]
    w = forked(**kw)
    begin, blocks = w.prefix_groups()
    assert (blocks > 0).any()
    g, o = prepared(w)
    out = g.decode_shared(partition_size=ps)
    ref = o.decode()
    torch.cuda.synchronize()
    H.assert_attention_close(H.out_to_double(out), ref, case + " " + route, w.io_dtype)
    assert int(g.dev_err.item()) == 0
    # the plain decode of the same batch agrees too
    out2 = g.decode(partition_size=ps)
    torch.cuda.synchronize()
    H.assert_attention_close(H.out_to_double(out2), ref, case + " plain", w.io_dtype)


def test_full_size_cow_layer():
    """The parallel-sampling layer at full size on the library's own route
    (the single pass, as the benchmark runs it), sampled rows against the
    oracle, and the split route agreeing with it everywhere."""
    w = W.cow_parallel_sampling_f16()
    g, o = prepared(w)
    out = g.decode_shared().clone()
    torch.cuda.synchronize()
    seqs = [0, 5, 6, 47, 90, 95]
    ref = o.decode(seqs)
    H.assert_attention_close(H.out_to_double(out)[seqs], ref, "cow full", w.io_dtype)
    assert int(g.dev_err.item()) == 0
    prev = B.pkv_testing_set_shared_prefix_path(2)
    try:
        split = g.decode_shared()
        torch.cuda.synchronize()
    finally:
        B.pkv_testing_set_shared_prefix_path(prev)
    # both routes are within 2e-3 + 2e-3 |ref| of the exact result; between
    # them, twice that
    a, b = H.out_to_double(out), H.out_to_double(split)
    assert np.all(np.abs(a - b) <= 2 * (H.ATOL + H.RTOL * np.abs(b)))
    assert int(g.dev_err.item()) == 0


def test_whole_context_shared_and_singletons(route):
    """A member whose context is exactly the prefix (nothing after it), groups
    of one, and a group whose entry says 0 blocks."""
    w = forked(num_heads=8, prompt_len=64, tail_hi=20)
    g, o = prepared(w)
    begin, blocks = w.prefix_groups()
    # shorten sample 1 of prompt 0 to the shared 4 blocks: it then has no
    # tokens past the prefix
    cl = w.context_lens.copy()
    cl[1] = 64
    g.context_lens.copy_(torch.from_numpy(cl))
    w2 = W.Workload(**{**w.__dict__, "context_lens": cl})
    ref = H.OracleRun(w2)
    ref.k_cache, ref.v_cache = o.k_cache, o.v_cache
    expect = ref.decode()
    # groups: [0, 6) with the prompt's 4 blocks, then six groups of one, the
    # first with an explicit 0
    grp = (np.array([0, 6, 7, 8, 9, 10, 11, 12], np.int32), np.array([4, 0, 0, 0, 0, 0, 0],
                                                                       np.int32))
    out = g.decode_shared(partition_size=32, groups=grp, max_group_size=6, max_prefix_blocks=4)
    torch.cuda.synchronize()
    H.assert_attention_close(H.out_to_double(out), expect, "whole-context prefix", w.io_dtype)
    assert int(g.dev_err.item()) == 0


def test_bad_group_entries_are_flagged(route):
    """A prefix longer than a member's context zeroes that member and flags
    PKV_DEVERR_CONTEXT; a member whose table differs inside the prefix flags
    PKV_DEVERR_PREFIX (its output is then not defined: the prefix kernel read
    the first member's block, whose unwritten slots hold the NaN sentinel);
    the other group is unaffected."""
    w = forked(num_heads=8, prompt_len=64, tail_hi=20)
    assert w.max_context_len >= 80
    g, o = prepared(w)
    # prefix of 5 blocks = 80 tokens: longer than the contexts of prompt 0's
    # samples that appended fewer than 16 tokens; the others hold their own
    # tail block at index 4, unlike the first sample
    short = [i for i in range(6) if w.context_lens[i] < 80]
    assert short and len(short) < 6
    grp = (np.array([0, 6, 12], np.int32), np.array([5, 4], np.int32))
    out = g.decode_shared(groups=grp, max_group_size=6, max_prefix_blocks=5)
    torch.cuda.synchronize()
    out = out.float().cpu()
    err = int(g.dev_err.item())
    assert err & B.PKV_DEVERR_CONTEXT and err & B.PKV_DEVERR_PREFIX
    for i in short:
        assert torch.all(out[i] == 0)
    # prompt 1's group stays correct
    ref = o.decode(list(range(6, 12)))
    H.assert_attention_close(out[6:12].double().numpy(), ref, "good group", w.io_dtype)
    # a member whose table differs in block 2 of the prefix
    g.dev_err.zero_()
    bt = w.block_tables.copy()
    bt[8, 2] = bt[8, 3]
    g.block_tables.copy_(torch.from_numpy(bt))
    g.decode_shared(groups=(np.array([0, 6, 12], np.int32), np.array([4, 4], np.int32)),
                    max_group_size=6, max_prefix_blocks=4)
    torch.cuda.synchronize()
    assert int(g.dev_err.item()) & B.PKV_DEVERR_PREFIX


def test_unusable_group_entry_zeroes_its_members(route):
    """A group whose prefix count exceeds max_prefix_blocks is flagged and its
    members' outputs are zero; the other group is unaffected."""
    w = forked(num_heads=8, prompt_len=64, tail_hi=20)
    g, o = prepared(w)
    out = g.decode_shared(groups=(np.array([0, 6, 12], np.int32), np.array([7, 4], np.int32)),
                          max_group_size=6, max_prefix_blocks=5)
    torch.cuda.synchronize()
    err = int(g.dev_err.item())
    assert err & B.PKV_DEVERR_PREFIX and err & B.PKV_DEVERR_CONTEXT
    got = out.float().cpu()
    assert torch.all(got[:6] == 0)
    ref = o.decode(list(range(6, 12)))
    H.assert_attention_close(got[6:12].double().numpy(), ref, "good group " + route, w.io_dtype)


def test_single_pass_wait_that_runs_out_is_flagged():
    """The single pass's bounded waits: with one poll per wait a wait runs
    out, PKV_DEVERR_TIMEOUT is set and the kernel returns; the next call, with
    the kernel's own limit, is correct."""
    w = forked(num_prompts=3)
    g, o = prepared(w)
    ref = o.decode()
    prev_path = B.pkv_testing_set_shared_prefix_path(1)
    prev = B.pkv_testing_set_decode_wait_limit(1)
    try:
        g.decode_shared()
        torch.cuda.synchronize()
        assert int(g.dev_err.item()) & B.PKV_DEVERR_TIMEOUT
    finally:
        B.pkv_testing_set_decode_wait_limit(prev)
    try:
        g.dev_err.zero_()
        out = g.decode_shared()
        torch.cuda.synchronize()
    finally:
        B.pkv_testing_set_shared_prefix_path(prev_path)
    assert int(g.dev_err.item()) == 0
    H.assert_attention_close(H.out_to_double(out), ref, "single pass after a time-out",
                             w.io_dtype)
