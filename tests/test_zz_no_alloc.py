"""The allocation-free decode entry point against the oracle and the regular one.

Some callers of this library cannot allocate device memory: an engine that has
reserved nearly all of the GPU's memory for its own KV-cache pool (a cudaMalloc
would fail), or a latency-critical path where cudaMalloc / cudaFree may
synchronise the device.  pkv_paged_attention_decode_static_ws serves them from
a static scratch array inside the library instead of a caller workspace.

Checked here, through the C ABI, with the output and the error word allocated
by the test before the calls (so the calls themselves allocate nothing):
its output matches the oracle within the parity tolerance of the other tests,
and pkv_paged_attention_decode on the same inputs within the same tolerance,
on calls in a row over a 16-bit and an E4M3 cache (each later call finds the
earlier call's partials still in the shared array); and a request larger than
the array is refused before any launch.  This file sorts last so that a run
stopping at the first failure has already run every other test.
"""
import ctypes

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


def _prepared(w):
    """The workload's cache on the device and, from the same inputs, the
    oracle's decode."""
    g = H.GpuRun(w)
    g.prefill()
    g.copy()
    g.step()
    o = H.OracleRun(w)
    o.prefill()
    o.copy()
    o.step()
    return g, o.decode()


def _check(g, oracle_out, partition_size, what):
    w = g.w
    # every device buffer the call touches exists before it
    out = torch.empty_like(g.q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = B.pkv_paged_attention_decode_static_ws(g.desc, g.q, g.block_tables, g.context_lens,
                                                 w.max_context_len, w.scale,
                                                 partition_size=partition_size, dev_err=err,
                                                 out=out)
    assert got.data_ptr() == out.data_ptr()
    ref = B.pkv_paged_attention_decode(g.desc, g.q, g.block_tables, g.context_lens,
                                       w.max_context_len, w.scale,
                                       partition_size=partition_size)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = H.out_to_double(out)
    H.assert_attention_close(got, oracle_out, what + " vs oracle", w.io_dtype)
    H.assert_attention_close(got, H.out_to_double(ref), what + " vs workspace decode",
                             w.io_dtype)


def test_static_scratch_decode_matches_oracle_on_calls_in_a_row():
    # first call: many partitions of an MHA layer; second: a grouped-head
    # layer with fewer, longer partitions; third: an E4M3 cache; fourth: the
    # first problem again, over the leftovers of the others
    a, a_ref = _prepared(W.opt13b_f16(num_seqs=8))
    _check(a, a_ref, 64, "static scratch, first call")
    b, b_ref = _prepared(W.llama2_70b_bf16_gqa(num_seqs=4))
    _check(b, b_ref, 256, "static scratch, second call")
    c, c_ref = _prepared(W.llama2_7b_fp8_long(num_seqs=3, lo=1024, hi=4096))
    _check(c, c_ref, 512, "static scratch, E4M3 call")
    _check(a, a_ref, 64, "static scratch, fourth call")


def test_request_beyond_the_static_scratch_is_refused():
    lib = B.load()
    # 64 sequences x 64 heads x 256 partitions of 16 tokens: far above 32 MiB of
    # partials.  Refused on the host before any pointer is used.
    desc = B.CacheDesc(0x10000, 0x20000, 1 << 20, 64, 16, 128, B.PKV_F16, 1.0, 1.0)
    need = B.pkv_decode_workspace_bytes(desc, 64, 64, 4096, 16)
    assert need > B.PKV_STATIC_SCRATCH_BYTES
    st = lib.pkv_paged_attention_decode_static_ws(
        ctypes.byref(desc), ctypes.c_void_p(0x1000), B.PKV_F16, 64, 64,
        ctypes.c_void_p(0x2000), 256, ctypes.c_void_p(0x3000), 4096, ctypes.c_float(0.1), 16,
        None, ctypes.c_void_p(0x4000), None)
    assert st == B.PKV_ERR_SCRATCH_LIMIT
    assert "static decode scratch" in B.pkv_status_string(st)
