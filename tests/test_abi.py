"""The C-ABI library builds, loads and exports every symbol include/pkv.h
declares; host-side argument checks reject bad calls before any launch.

These run without a GPU: every call below fails a host check (or is a pure
host query), so nothing is launched and no pointer is dereferenced.
"""
import ctypes

import pytest

from paged_kv_cache_130_gb300 import binding as B
from paged_kv_cache_130_gb300 import build as pkv_build


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return B.load()


def _desc(**kw):
    d = dict(k_cache=0x10000, v_cache=0x20000, num_blocks=64, num_kv_heads=8, block_size=16,
             head_dim=128, cache_dtype=B.PKV_F16, k_scale=1.0, v_scale=1.0)
    d.update(kw)
    return B.CacheDesc(**d)


def test_every_declared_symbol_is_exported(lib):
    names = B.header_functions()
    assert {"pkv_kv_append", "pkv_copy_blocks", "pkv_paged_attention_decode",
            "pkv_paged_attention_partitions", "pkv_lse_reduce", "pkv_decode_workspace_bytes",
            "pkv_decode_partition_size", "pkv_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert B.pkv_status_string(0) == "ok"
    assert "workspace" in B.pkv_status_string(B.PKV_ERR_WORKSPACE)
    assert B.pkv_status_string(99) == "unknown status"


def test_partition_size_and_workspace(lib):
    d = _desc()
    # few items: split at 256 KiB of fp16 K+V (512 tokens) per KV head
    assert B.pkv_decode_partition_size(d, 4, 8, 3000, 0) == 512
    # grouped heads, between one and two waves of (sequence, KV head) items
    # (W = 3 x 152 SMs without a GPU): the contexts above 3/4 of the longest
    # are cut in two; two waves or more: one partition per context
    assert B.pkv_decode_partition_size(d, 64, 64, 3000, 0) == 2256
    assert B.pkv_decode_partition_size(d, 120, 64, 3000, 0) == 3008
    # grouped heads, fewer items: 1 MiB of K+V per partition (2048 tokens)
    assert B.pkv_decode_partition_size(d, 16, 64, 3000, 0) == 2048
    # many single-head items over short contexts: one partition per context
    d40 = _desc(num_kv_heads=40)
    assert B.pkv_decode_partition_size(d40, 32, 40, 1398, 0) == 1408
    assert B.pkv_decode_partition_size(d40, 32, 40, 9000, 0) == 512       # too long
    assert B.pkv_decode_partition_size(d40, 200, 40, 1398, 0) == 512      # too many to rank
    assert B.pkv_decode_partition_size(d, 4, 8, 3000, 64) == 64           # as requested
    f8 = _desc(cache_dtype=B.PKV_FP8_E4M3, block_size=32)
    assert B.pkv_decode_partition_size(f8, 4, 8, 30000, 0) == 1024
    # a context within one partition needs no workspace
    assert B.pkv_decode_workspace_bytes(d, 4, 8, 512, 0) == 0
    s, h, p, dim = 3, 8, 2, 128
    ml = -(-4 * s * h * p // 256) * 256
    want = 2 * ml + -(-4 * s * h * p * dim // 256) * 256
    assert B.pkv_decode_workspace_bytes(d, s, h, 700, 0) == want


def _append(lib, desc, k=0x1000, v=0x2000, in_dtype=B.PKV_F16, slots=0x3000, n=4):
    return lib.pkv_kv_append(ctypes.byref(desc), ctypes.c_void_p(k), ctypes.c_void_p(v),
                             in_dtype, ctypes.c_void_p(slots), n, None, None)


def test_append_host_checks(lib):
    assert _append(lib, _desc(head_dim=96)) == B.PKV_ERR_UNSUPPORTED
    assert _append(lib, _desc(block_size=12)) == B.PKV_ERR_UNSUPPORTED
    assert _append(lib, _desc(k_cache=0x10001)) == B.PKV_ERR_INVALID_ARG
    assert _append(lib, _desc(), k=0x1004) == B.PKV_ERR_INVALID_ARG
    assert _append(lib, _desc(), slots=0) == B.PKV_ERR_INVALID_ARG
    assert _append(lib, _desc(), n=-1) == B.PKV_ERR_INVALID_ARG
    assert _append(lib, _desc(), in_dtype=B.PKV_FP8_E4M3) == B.PKV_ERR_INVALID_ARG
    assert _append(lib, _desc(cache_dtype=B.PKV_BF16)) == B.PKV_ERR_UNSUPPORTED
    assert _append(lib, _desc(cache_dtype=B.PKV_FP8_E4M3, k_scale=0.0)) == B.PKV_ERR_INVALID_ARG
    assert _append(lib, _desc(), n=0) == B.PKV_OK                 # no-op, nothing launched


def _decode(lib, desc, q_dtype=B.PKV_F16, S=2, H=8, bt=0x4000, mb=4, ctx=0x5000, maxctx=64,
            part=0, ws=None, ws_bytes=0, out=0x6000, q=0x7000, fn="pkv_paged_attention_decode"):
    return getattr(lib, fn)(ctypes.byref(desc), ctypes.c_void_p(q), q_dtype, S, H,
                            ctypes.c_void_p(bt), mb, ctypes.c_void_p(ctx), maxctx,
                            ctypes.c_float(0.1), part, ctypes.c_void_p(ws), ws_bytes, None,
                            ctypes.c_void_p(out), None)


@pytest.mark.parametrize("fn", ["pkv_paged_attention_decode", "pkv_paged_attention_partitions"])
def test_decode_host_checks(lib, fn):
    d = _desc()
    assert _decode(lib, d, H=12, fn=fn) == B.PKV_ERR_INVALID_ARG          # 12 % 8 != 0
    assert _decode(lib, d, q_dtype=B.PKV_BF16, fn=fn) == B.PKV_ERR_UNSUPPORTED
    assert _decode(lib, d, part=24, fn=fn) == B.PKV_ERR_INVALID_ARG       # not a multiple of 16
    assert _decode(lib, d, out=0x6002, fn=fn) == B.PKV_ERR_INVALID_ARG
    assert _decode(lib, d, ctx=0, fn=fn) == B.PKV_ERR_INVALID_ARG
    assert _decode(lib, _desc(head_dim=80), fn=fn) == B.PKV_ERR_UNSUPPORTED
    # two partitions need a workspace
    assert _decode(lib, d, maxctx=700, fn=fn) == B.PKV_ERR_WORKSPACE
    assert _decode(lib, d, maxctx=700, ws=0x100010, ws_bytes=1 << 20, fn=fn) == \
        B.PKV_ERR_WORKSPACE                                              # misaligned
    assert _decode(lib, d, maxctx=700, ws=0x100000, ws_bytes=16, fn=fn) == B.PKV_ERR_WORKSPACE
    assert _decode(lib, d, S=0, fn=fn) == B.PKV_OK                       # nothing to do


def test_copy_and_reduce_host_checks(lib):
    arr = (B.CacheDesc * 2)(_desc(), _desc(num_blocks=65))
    assert lib.pkv_copy_blocks(arr, 2, ctypes.c_void_p(0x1000), 3, None, None) == \
        B.PKV_ERR_INVALID_ARG                                            # layers differ
    arr = (B.CacheDesc * 1)(_desc())
    assert lib.pkv_copy_blocks(arr, 1, None, 3, None, None) == B.PKV_ERR_INVALID_ARG
    assert lib.pkv_copy_blocks(arr, 1, None, 0, None, None) == B.PKV_OK
    assert lib.pkv_lse_reduce(2, 8, 96, ctypes.c_void_p(0x1000), 100, 32, None, 0, 0,
                              ctypes.c_void_p(0x2000), None) == B.PKV_ERR_INVALID_ARG
    assert lib.pkv_lse_reduce(2, 8, 128, ctypes.c_void_p(0x1000), 100, 32, None, 0, 0,
                              ctypes.c_void_p(0x2000), None) == B.PKV_ERR_WORKSPACE


def _shared(lib, desc, S=2, H=8, maxctx=64, ng=1, gb=0x8000, gp=0x9000, mgs=2, mpb=2,
            part=0, ws=None, ws_bytes=0, q_dtype=B.PKV_F16):
    return lib.pkv_paged_attention_decode_shared_prefix(
        ctypes.byref(desc), ctypes.c_void_p(0x7000), q_dtype, S, H, ctypes.c_void_p(0x4000), 4,
        ctypes.c_void_p(0x5000), maxctx, ng, ctypes.c_void_p(gb), ctypes.c_void_p(gp), mgs, mpb,
        ctypes.c_float(0.1), part, ctypes.c_void_p(ws), ws_bytes, None, ctypes.c_void_p(0x6000),
        None)


def test_shared_prefix_host_checks(lib):
    d = _desc()
    # four more partials per row than the plain decode (the prefix pieces)
    plain = B.pkv_decode_workspace_bytes(d, 4, 8, 3000, 512)
    shared = B.pkv_shared_prefix_workspace_bytes(d, 4, 8, 3000, 512)
    s, h, p, dim = 4, 8, 6 + 4, 128
    ml = -(-4 * s * h * p // 256) * 256
    assert shared == 2 * ml + -(-4 * s * h * p * dim // 256) * 256 and shared > plain
    # a context within one partition still needs the workspace with a prefix
    assert B.pkv_shared_prefix_workspace_bytes(d, 4, 8, 512, 512) > 0
    assert _shared(lib, _desc(cache_dtype=B.PKV_FP8_E4M3, block_size=32)) == \
        B.PKV_ERR_UNSUPPORTED
    assert _shared(lib, d, q_dtype=B.PKV_BF16) == B.PKV_ERR_UNSUPPORTED    # mixed types
    assert _shared(lib, d, mpb=5) == B.PKV_ERR_INVALID_ARG     # 5 * 16 > max_context_len 64
    assert _shared(lib, d, mpb=5, maxctx=80) == B.PKV_ERR_INVALID_ARG      # > 4 table entries
    assert _shared(lib, d, gb=0) == B.PKV_ERR_INVALID_ARG
    assert _shared(lib, d, ng=3) == B.PKV_ERR_INVALID_ARG      # more groups than sequences
    assert _shared(lib, d, mgs=0) == B.PKV_ERR_INVALID_ARG
    assert _shared(lib, d) == B.PKV_ERR_WORKSPACE              # the prefix needs partials
    assert _shared(lib, d, S=0) == B.PKV_OK


def test_swap_host_checks(lib):
    d = _desc()
    arr = (B.CacheDesc * 1)(d)
    other = (B.CacheDesc * 1)(_desc(head_dim=64))
    assert lib.pkv_swap_blocks(None, arr, 1, ctypes.c_void_p(0x1000), 1, None, None) == \
        B.PKV_ERR_INVALID_ARG
    assert lib.pkv_swap_blocks(arr, arr, 0, ctypes.c_void_p(0x1000), 1, None, None) == \
        B.PKV_ERR_INVALID_ARG
    assert lib.pkv_swap_blocks(arr, other, 1, ctypes.c_void_p(0x1000), 1, None, None) == \
        B.PKV_ERR_INVALID_ARG                                            # shapes differ
    assert lib.pkv_swap_blocks(arr, arr, 1, None, 0, None, None) == B.PKV_OK
    # a pointer CUDA does not know is refused before any launch
    assert lib.pkv_swap_blocks(arr, arr, 1, ctypes.c_void_p(0x1000), 2, None, None) == \
        B.PKV_ERR_INVALID_ARG


def test_block_hash_host_checks(lib):
    f = lib.pkv_block_hashes
    p = ctypes.c_void_p
    assert f(p(0x1000), p(0x2000), 2, 10, 12, None, p(0x3000), 1, p(0x4000), None, None) == \
        B.PKV_ERR_UNSUPPORTED                                            # block size 12
    assert f(p(0x1000), None, 2, 10, 16, None, p(0x3000), 1, p(0x4000), None, None) == \
        B.PKV_ERR_INVALID_ARG
    assert f(p(0x1000), p(0x2000), 2, 10, 16, None, p(0x3000), 1, p(0x4004), None, None) == \
        B.PKV_ERR_INVALID_ARG                                            # misaligned output
    assert f(None, None, 0, 0, 16, None, None, 0, None, None, None) == B.PKV_OK
