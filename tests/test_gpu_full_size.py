"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (same workloads, same partition sizes).

The oracle computes four of the five layers completely: every cache byte after
prefill, copy-on-write and the step's append is compared, and every output
element.  For the long-context FP8 layer (2.7 GB of cache) it computes three
sampled sequences one by one: all bytes of their blocks and all their outputs.
"""
import numpy as np
import pytest
import torch

import harness as H
from paged_kv_cache_130_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    H.build_library()


@pytest.mark.parametrize("name", ["opt13b_f16", "llama2_70b_bf16_gqa",
                                  "cow_parallel_sampling_f16"])
def test_full_size_layer(name):
    w = W.make(name)
    g = H.GpuRun(w)
    o = H.OracleRun(w)
    H.prefill_both(w, g, o)
    g.copy()
    o.copy()
    g.step()
    o.step()
    torch.cuda.synchronize()
    assert np.array_equal(H.to_bits(g.k_cache), o.k_cache), "K cache bytes"
    assert np.array_equal(H.to_bits(g.v_cache), o.v_cache), "V cache bytes"
    out = g.decode()
    torch.cuda.synchronize()
    ref = o.decode()
    H.assert_attention_close(H.out_to_double(out), ref, name, w.io_dtype)
    assert int(g.dev_err.item()) == 0
    del g
    torch.cuda.empty_cache()


def test_full_size_fp8_long_context_sampled():
    w = W.llama2_7b_fp8_long()
    seqs = [0, 7, w.num_seqs - 1]
    g = H.GpuRun(w)
    o = H.OracleRun(w)
    H.prefill_both(w, g, o, only=seqs)
    g.step()
    o.step()
    out = g.decode()
    torch.cuda.synchronize()
    assert int(g.dev_err.item()) == 0
    for s in seqs:
        nblk = -(-int(w.context_lens[s]) // w.block_size)
        blocks = torch.from_numpy(w.block_tables[s, :nblk].astype(np.int64)).cuda()
        gk = H.to_bits(g.k_cache.index_select(0, blocks))
        gv = H.to_bits(g.v_cache.index_select(0, blocks))
        idx = w.block_tables[s, :nblk]
        assert np.array_equal(gk, o.k_cache[idx]), "K bytes of sequence %d" % s
        assert np.array_equal(gv, o.v_cache[idx]), "V bytes of sequence %d" % s
    ref = o.decode(seqs)
    H.assert_attention_close(H.out_to_double(out)[seqs], ref, "fp8 sampled", w.io_dtype)
    del g
    torch.cuda.empty_cache()
