"""Causal prefill attention over the paged cache (tensor-core kernel) against
the oracle: |gpu - oracle| <= 2e-3 + 2e-3 |oracle| (plus half an ulp of the
output type), every new token of small batches, sampled rows of the
full-size workloads.  The prompt's K/V are appended with kv_append first and
checked byte for byte."""
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


def prepared(w):
    g = H.GpuRun(w)
    o = H.OracleRun(w)
    for r in (g, o):
        r.prefill()
        r.step()
    torch.cuda.synchronize()
    assert np.array_equal(H.to_bits(g.k_cache), o.k_cache), "K bytes"
    assert np.array_equal(H.to_bits(g.v_cache), o.v_cache), "V bytes"
    return g, o


SHAPES = [
    # dtype, heads, kv heads, D, block, new tokens, cached tokens
    (W.BF16, 4, 4, 128, 16, [70, 1, 129, 64], [0, 0, 0, 0]),
    (W.F16, 4, 4, 128, 16, [70, 1, 129, 64], [0, 0, 0, 0]),
    (W.BF16, 8, 2, 64, 32, [33, 100, 7], [40, 0, 200]),
    (W.F16, 16, 2, 128, 8, [17, 65, 3], [5, 130, 64]),
    (W.BF16, 16, 1, 64, 16, [9, 20], [100, 0]),           # 16 heads per KV head
    (W.F16, 64, 1, 64, 16, [3, 2], [31, 0]),              # one token per CTA
    (W.BF16, 6, 2, 128, 16, [50, 23], [10, 77]),          # 3 heads per KV head: 21 tokens
]


@pytest.mark.parametrize("i", range(len(SHAPES)))
def test_prefill_shapes(i):
    dt, h, hkv, d, bs, new, cached = SHAPES[i]
    w = W._prompts("prefill_case", 20 + i, dt, h, hkv, d, bs, new, cached)
    g, o = prepared(w)
    out = g.prefill_attention()
    torch.cuda.synchronize()
    ref = o.prefill_attention()
    H.assert_attention_close(H.out_to_double(out), ref, "prefill %d" % i, dt)
    assert int(g.dev_err.item()) == 0


@pytest.mark.parametrize("name,rows", [("prefill_llama2_7b_bf16", 48),
                                       ("prefill_llama2_70b_gqa_chunked_bf16", 24)])
def test_prefill_full_size_sampled(name, rows):
    w = W.make(name)
    g, o = prepared(w)
    out = g.prefill_attention()
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    cu = w.cu_seqlens_q
    pick = set(rng.choice(w.total_q, rows, replace=False).tolist())
    pick |= {int(cu[s]) for s in range(w.num_seqs)} | {int(cu[s + 1]) - 1
                                                        for s in range(w.num_seqs)}
    pick = np.array(sorted(pick))
    ref = o.prefill_attention(pick)
    H.assert_attention_close(H.out_to_double(out)[pick], ref, name, w.io_dtype)
    assert int(g.dev_err.item()) == 0


def test_prefill_first_token_is_its_v_exactly():
    w = W._prompts("prefill_first", 31, W.BF16, 8, 8, 128, 16, [40, 17], [0, 0])
    g, o = prepared(w)
    out = H.to_bits(g.prefill_attention())
    torch.cuda.synchronize()
    k, v = w.step_values()
    cu = w.cu_seqlens_q
    for s in range(2):
        # row cu[s] attends to its own token only: out = v exactly
        assert np.array_equal(out[cu[s]], v[cu[s]])


def test_prefill_bad_lengths_are_flagged():
    w = W._prompts("prefill_bad", 32, W.F16, 4, 4, 64, 16, [20, 30], [0, 10])
    g, o = prepared(w)
    cl = w.context_lens.copy()
    cl[0] = 10                                   # fewer cached tokens than new ones
    g.context_lens.copy_(torch.from_numpy(cl))
    out = g.prefill_attention()
    torch.cuda.synchronize()
    assert int(g.dev_err.item()) & B.PKV_DEVERR_CONTEXT
    assert torch.all(out[:20] == 0)
    ref = o.prefill_attention(np.arange(20, 50))
    H.assert_attention_close(H.out_to_double(out)[20:50], ref, "good sequence", W.F16)


def test_prefill_grid_larger_than_the_prompts():
    """max_q_len above every prompt: the extra work items find no rows and the
    output is the same."""
    w = W._prompts("prefill_wide", 33, W.BF16, 8, 2, 128, 16, [40, 300, 129], [0, 60, 7])
    g, o = prepared(w)
    cu = torch.from_numpy(w.cu_seqlens_q).to(g.device)
    out = B.pkv_paged_attention_prefill(g.desc, g.q, cu, 4 * w.max_q_len + 3, g.block_tables,
                                        g.context_lens, w.max_context_len, w.scale,
                                        dev_err=g.dev_err)
    torch.cuda.synchronize()
    H.assert_attention_close(H.out_to_double(out), o.prefill_attention(), "wide grid", W.BF16)
    assert int(g.dev_err.item()) == 0


def test_prefill_bad_block_id_is_flagged_and_contained():
    """A negative block id in one table: PKV_DEVERR_BLOCK_ID is raised, rows
    whose keys all come before that block and the other sequences keep the
    exact results, and no output is NaN (the block reads as zeros)."""
    w = W._prompts("prefill_badblock", 34, W.F16, 4, 4, 64, 16, [300, 90], [0, 0])
    g, o = prepared(w)
    bt = w.block_tables.copy()
    bad = 10                                      # keys 160..175 of sequence 0
    bt[0, bad] = -3
    g.block_tables.copy_(torch.from_numpy(bt))
    out = g.prefill_attention()
    torch.cuda.synchronize()
    assert int(g.dev_err.item()) & B.PKV_DEVERR_BLOCK_ID
    got = H.out_to_double(out)
    assert not np.isnan(got).any()
    cu = w.cu_seqlens_q
    keep = np.r_[np.arange(cu[0], cu[0] + bad * 16), np.arange(cu[1], cu[2])]
    H.assert_attention_close(got[keep], o.prefill_attention(keep), "rows before the bad block",
                             W.F16)
