"""The streaming decode kernel's bounded waits and its work-counter slots.

Every mbarrier wait of the streaming decode kernel is bounded: when a wait
runs out, the kernel sets PKV_DEVERR_TIMEOUT, stops waiting everywhere, lets
the bulk copies it started land, and returns, so that the CUDA context stays
usable.  These tests make the waits run out on purpose, through the library's
testing setting of the wait limit (one poll per wait), and then check that
the flag is set and that a following normal decode is correct.  Nothing here
faults, traps or hangs: the waits that run out are bounded, and the drain of
copies in flight keeps the kernel's full limit.

The kernel hands out work from one of 1024 device counter slots, taken in turn
per launch (a captured graph keeps its slot).  The second test runs more than
1024 launches on one stream with graph replays between them, so that slots are
reused back to back, and checks that every result is the same and that no
launch flags PKV_DEVERR_SCHED.
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
    B.pkv_testing_set_decode_wait_limit(0)


def _prepared(w):
    g = H.GpuRun(w)
    g.prefill()
    g.copy()
    g.step()
    o = H.OracleRun(w)
    o.prefill()
    o.copy()
    o.step()
    return g, o.decode()


def _decode(g, partition_size):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = B.pkv_paged_attention_decode(g.desc, g.q, g.block_tables, g.context_lens,
                                       g.w.max_context_len, g.w.scale,
                                       partition_size=partition_size, dev_err=err)
    torch.cuda.synchronize()
    return out, int(err.item())


@pytest.mark.parametrize("name,ps", [("opt13b_f16", 64), ("opt13b_f16", 0),
                                     ("llama2_7b_fp8_long", 512)])
def test_wait_that_runs_out_flags_timeout_and_the_next_decode_is_correct(name, ps):
    w = (W.opt13b_f16(num_seqs=8) if name == "opt13b_f16"
         else W.llama2_7b_fp8_long(num_seqs=3, lo=1024, hi=4096))
    g, ref = _prepared(w)
    prev = B.pkv_testing_set_decode_wait_limit(1)
    try:
        _, err = _decode(g, ps)
    finally:
        B.pkv_testing_set_decode_wait_limit(prev)
    assert err & B.PKV_DEVERR_TIMEOUT, "a one-poll wait limit did not run out (err=%d)" % err
    # the context is usable and the next call, with the kernel's own limit, is right
    out, err = _decode(g, ps)
    assert err == 0
    H.assert_attention_close(H.out_to_double(out), ref, "after a time-out", w.io_dtype)


def test_scheduler_slots_reused_back_to_back_on_one_stream():
    w = W.opt13b_f16(num_seqs=4)
    g = H.GpuRun(w)
    g.prefill()
    g.step()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(g.q)

    def call():
        B.pkv_paged_attention_decode(g.desc, g.q, g.block_tables, g.context_lens,
                                     w.max_context_len, w.scale, dev_err=err, out=out)

    call()
    torch.cuda.synchronize()
    first = out.clone()
    # a captured decode keeps the slot it took at capture for every replay
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    mismatches = 0
    for i in range(1100):
        out.zero_()
        if i % 50 == 0:
            graph.replay()
        else:
            call()
        if i % 10 == 0 or 1015 <= i <= 1035:
            torch.cuda.synchronize()
            mismatches += int(not torch.equal(out.view(torch.int16), first.view(torch.int16)))
    torch.cuda.synchronize()
    assert mismatches == 0
    assert int(err.item()) == 0, "dev_err %d" % int(err.item())
    np.testing.assert_array_equal(H.to_bits(out), H.to_bits(first))
