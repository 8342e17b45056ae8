"""Thin ctypes binding of libpkv.so (include/pkv.h).

Argument marshalling only: tensors become device pointers, torch dtypes become
pkv_dtype codes, the stream defaults to torch's current stream, and a non-zero
status raises :class:`PkvError`.  Every step of the computation runs in the
library's CUDA kernels; there is no other path.  When the library has not been
built the first call raises.

The functions carry the C names.  Caches are described by :class:`CacheDesc`
(``pkv_cache_desc``); :func:`cache_desc` fills one from two torch tensors.
"""
import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpkv.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "pkv.h")

PKV_F16, PKV_BF16, PKV_FP8_E4M3 = 0, 1, 2
PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE, PKV_ERR_CUDA = range(5)
PKV_ERR_SCRATCH_LIMIT = 5
PKV_STATIC_SCRATCH_BYTES = 32 << 20
PKV_DEVERR_SLOT, PKV_DEVERR_BLOCK_ID, PKV_DEVERR_CONTEXT, PKV_DEVERR_COPY_PAIR = 1, 2, 4, 8
PKV_DEVERR_TIMEOUT = 16
PKV_DEVERR_PREFIX = 32
PKV_DEVERR_SCHED = 64


class PkvError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, pkv_status_string(status), status))


class CacheDesc(ctypes.Structure):
    _fields_ = [("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int64), ("num_kv_heads", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("cache_dtype", ctypes.c_int32), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float)]


_lib = None


def library_path():
    return LIB_PATH


def load():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libpkv.so is not built (%s); run paged_kv_cache_130_gb300.build.build()"
                           % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    dp = ctypes.POINTER(CacheDesc)
    sigs = {
        "pkv_status_string": (ctypes.c_char_p, [i32]),
        "pkv_kv_append": (i32, [dp, vp, vp, i32, vp, i64, vp, vp]),
        "pkv_copy_blocks": (i32, [dp, i32, vp, i64, vp, vp]),
        "pkv_decode_partition_size": (i32, [dp, i32, i32, i32, i32]),
        "pkv_decode_workspace_bytes": (ctypes.c_size_t, [dp, i32, i32, i32, i32]),
        "pkv_paged_attention_decode": (i32, [dp, vp, i32, i32, i32, vp, i32, vp, i32, f32, i32,
                                             vp, ctypes.c_size_t, vp, vp, vp]),
        "pkv_paged_attention_partitions": (i32, [dp, vp, i32, i32, i32, vp, i32, vp, i32, f32,
                                                 i32, vp, ctypes.c_size_t, vp, vp, vp]),
        "pkv_lse_reduce": (i32, [i32, i32, i32, vp, i32, i32, vp, ctypes.c_size_t, i32, vp, vp]),
        "pkv_paged_attention_decode_static_ws": (i32, [dp, vp, i32, i32, i32, vp, i32, vp, i32,
                                                       f32, i32, vp, vp, vp]),
        "pkv_shared_prefix_workspace_bytes": (ctypes.c_size_t, [dp, i32, i32, i32, i32]),
        "pkv_swap_blocks": (i32, [dp, dp, i32, vp, i64, vp, vp]),
        "pkv_block_hashes": (i32, [vp, vp, i32, i64, i32, vp, vp, i64, vp, vp, vp]),
        "pkv_paged_attention_prefill": (i32, [dp, vp, i32, i32, i32, vp, i32, i32, vp, i32,
                                              vp, i32, f32, vp, vp, vp]),
        "pkv_paged_attention_decode_shared_prefix": (i32, [dp, vp, i32, i32, i32, vp, i32, vp,
                                                           i32, i32, vp, vp, i32, i32, f32, i32,
                                                           vp, ctypes.c_size_t, vp, vp, vp]),
        "pkv_testing_set_decode_wait_limit": (ctypes.c_uint32, [ctypes.c_uint32]),
        "pkv_testing_set_shared_prefix_path": (i32, [i32]),
        "pkv_testing_stream_copy": (i32, [vp, vp, i64, vp]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def header_functions():
    """Names of the functions include/pkv.h declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


# ------------------------------------------------------------------ helpers

def dtype_code(t):
    if t == torch.float16:
        return PKV_F16
    if t == torch.bfloat16:
        return PKV_BF16
    if t in (torch.uint8, getattr(torch, "float8_e4m3fn", None)):
        return PKV_FP8_E4M3
    raise TypeError("unsupported element type %s" % t)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(status, where):
    if status != PKV_OK:
        raise PkvError(status, where)


def _dense(t, name):
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t


def cache_desc(k_cache, v_cache, k_scale=1.0, v_scale=1.0):
    """Descriptor of one layer's caches, each [num_blocks, num_kv_heads, block_size, head_dim]."""
    _dense(k_cache, "k_cache")
    _dense(v_cache, "v_cache")
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype or k_cache.dim() != 4:
        raise ValueError("k_cache and v_cache must be alike, 4-D")
    nb, hkv, bs, d = k_cache.shape
    return CacheDesc(k_cache.data_ptr(), v_cache.data_ptr(), nb, hkv, bs, d,
                     dtype_code(k_cache.dtype), float(k_scale), float(v_scale))


# ------------------------------------------------------------------ entry points

def pkv_status_string(status):
    return load().pkv_status_string(int(status)).decode()


def pkv_kv_append(cache, k, v, slot_mapping, dev_err=None, stream=None):
    _dense(k, "k")
    _dense(v, "v")
    _dense(slot_mapping, "slot_mapping")
    if slot_mapping.dtype != torch.int64 or k.shape != v.shape:
        raise ValueError("slot_mapping must be int64 and k, v alike")
    _check(load().pkv_kv_append(ctypes.byref(cache), _ptr(k), _ptr(v), dtype_code(k.dtype),
                                _ptr(slot_mapping), slot_mapping.numel(), _ptr(dev_err),
                                _stream(stream)), "pkv_kv_append")


def pkv_copy_blocks(caches, block_pairs, dev_err=None, stream=None):
    if isinstance(caches, CacheDesc):
        caches = [caches]
    arr = (CacheDesc * len(caches))(*caches)
    _dense(block_pairs, "block_pairs")
    if block_pairs.dtype != torch.int64:
        raise ValueError("block_pairs must be int64 [n, 2]")
    n = block_pairs.numel() // 2
    _check(load().pkv_copy_blocks(arr, len(caches), _ptr(block_pairs), n, _ptr(dev_err),
                                  _stream(stream)), "pkv_copy_blocks")


def pkv_decode_partition_size(cache, num_seqs, num_heads, max_context_len, requested=0):
    return int(load().pkv_decode_partition_size(ctypes.byref(cache), int(num_seqs),
                                                int(num_heads), int(max_context_len),
                                                int(requested)))


def pkv_decode_workspace_bytes(cache, num_seqs, num_heads, max_context_len, partition_size=0):
    return int(load().pkv_decode_workspace_bytes(ctypes.byref(cache), num_seqs, num_heads,
                                                 max_context_len, partition_size))


def _decode_common(fn, where, cache, q, block_tables, context_lens, max_context_len, scale,
                   partition_size, workspace, dev_err, out, stream):
    _dense(q, "q")
    _dense(block_tables, "block_tables")
    _dense(context_lens, "context_lens")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    s, h, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    need = pkv_decode_workspace_bytes(cache, s, h, max_context_len, partition_size)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(fn(ctypes.byref(cache), _ptr(q), dtype_code(q.dtype), s, h, _ptr(block_tables),
              block_tables.shape[1], _ptr(context_lens), int(max_context_len), float(scale),
              int(partition_size), _ptr(workspace), ws_bytes, _ptr(dev_err), _ptr(out),
              _stream(stream)), where)
    return out


def pkv_paged_attention_decode(cache, q, block_tables, context_lens, max_context_len, scale,
                               partition_size=0, workspace=None, dev_err=None, out=None,
                               stream=None):
    return _decode_common(load().pkv_paged_attention_decode, "pkv_paged_attention_decode",
                          cache, q, block_tables, context_lens, max_context_len, scale,
                          partition_size, workspace, dev_err, out, stream)


def pkv_paged_attention_partitions(cache, q, block_tables, context_lens, max_context_len, scale,
                                   partition_size=0, workspace=None, dev_err=None, out=None,
                                   stream=None):
    return _decode_common(load().pkv_paged_attention_partitions,
                          "pkv_paged_attention_partitions", cache, q, block_tables,
                          context_lens, max_context_len, scale, partition_size, workspace,
                          dev_err, out, stream)


def pkv_lse_reduce(num_seqs, num_heads, head_dim, context_lens, max_context_len, partition_size,
                   workspace, out, stream=None):
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(load().pkv_lse_reduce(num_seqs, num_heads, head_dim, _ptr(context_lens),
                                 int(max_context_len), int(partition_size), _ptr(workspace),
                                 ws_bytes, dtype_code(out.dtype), _ptr(out), _stream(stream)),
           "pkv_lse_reduce")
    return out


def pkv_paged_attention_decode_static_ws(cache, q, block_tables, context_lens, max_context_len,
                                         scale, partition_size=0, dev_err=None, out=None,
                                         stream=None):
    """Decode without a caller workspace: for callers that cannot allocate
    device memory (an engine that has reserved the GPU's memory for its own
    cache pool, or a latency-critical path where cudaMalloc may synchronise).
    The partials live in the library's static 32 MiB device array; calls that
    overlap on the GPU race on it, so keep them on one stream."""
    _dense(q, "q")
    _dense(block_tables, "block_tables")
    _dense(context_lens, "context_lens")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    s, h, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    _check(load().pkv_paged_attention_decode_static_ws(
        ctypes.byref(cache), _ptr(q), dtype_code(q.dtype), s, h, _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), int(max_context_len), float(scale),
        int(partition_size), _ptr(dev_err), _ptr(out), _stream(stream)),
        "pkv_paged_attention_decode_static_ws")
    return out


def pkv_testing_set_decode_wait_limit(tries):
    """Polls per bounded wait of the streaming decode kernel for later decode
    calls (0: the kernel's own limit); a testing aid.  Returns the previous
    setting."""
    return int(load().pkv_testing_set_decode_wait_limit(int(tries)))


def pkv_testing_set_shared_prefix_path(path):
    """Route of later shared-prefix decode calls (0: the library's choice,
    1: the single pass, 2: prefix kernel + partitions + reduce); a testing
    aid.  Returns the previous setting."""
    r = int(load().pkv_testing_set_shared_prefix_path(int(path)))
    if r < 0:
        raise ValueError("path must be 0, 1 or 2")
    return r


def pkv_shared_prefix_workspace_bytes(cache, num_seqs, num_heads, max_context_len,
                                      partition_size=0):
    return int(load().pkv_shared_prefix_workspace_bytes(ctypes.byref(cache), num_seqs,
                                                        num_heads, max_context_len,
                                                        partition_size))


def pkv_paged_attention_decode_shared_prefix(cache, q, block_tables, context_lens,
                                             max_context_len, group_begin, group_prefix_blocks,
                                             max_group_size, max_prefix_blocks, scale,
                                             partition_size=0, workspace=None, dev_err=None,
                                             out=None, stream=None):
    """Decode where the sequences [group_begin[i], group_begin[i+1]) share their
    first group_prefix_blocks[i] blocks (int32 device tensors); the two
    max_* arguments are host upper bounds."""
    _dense(q, "q")
    _dense(block_tables, "block_tables")
    _dense(context_lens, "context_lens")
    _dense(group_begin, "group_begin")
    _dense(group_prefix_blocks, "group_prefix_blocks")
    for t, name in ((block_tables, "block_tables"), (context_lens, "context_lens"),
                    (group_begin, "group_begin"), (group_prefix_blocks, "group_prefix_blocks")):
        if t.dtype != torch.int32:
            raise ValueError("%s must be int32" % name)
    num_groups = group_prefix_blocks.numel()
    if group_begin.numel() != num_groups + 1:
        raise ValueError("group_begin needs num_groups + 1 entries")
    s, h, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    need = pkv_shared_prefix_workspace_bytes(cache, s, h, max_context_len, partition_size)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().pkv_paged_attention_decode_shared_prefix(
        ctypes.byref(cache), _ptr(q), dtype_code(q.dtype), s, h, _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), int(max_context_len), num_groups,
        _ptr(group_begin), _ptr(group_prefix_blocks), int(max_group_size),
        int(max_prefix_blocks), float(scale), int(partition_size), _ptr(workspace), ws_bytes,
        _ptr(dev_err), _ptr(out), _stream(stream)), "pkv_paged_attention_decode_shared_prefix")
    return out


def pkv_paged_attention_prefill(cache, q, cu_seqlens_q, max_q_len, block_tables, context_lens,
                                max_context_len, scale, dev_err=None, out=None, stream=None):
    """Causal prefill of q [total_q, num_heads, head_dim]: sequence s owns rows
    [cu_seqlens_q[s], cu_seqlens_q[s+1]), the last tokens of its context."""
    _dense(q, "q")
    for t, name in ((cu_seqlens_q, "cu_seqlens_q"), (block_tables, "block_tables"),
                    (context_lens, "context_lens")):
        _dense(t, name)
        if t.dtype != torch.int32:
            raise ValueError("%s must be int32" % name)
    total, h, d = q.shape
    num_seqs = context_lens.numel()
    if cu_seqlens_q.numel() != num_seqs + 1:
        raise ValueError("cu_seqlens_q needs num_seqs + 1 entries")
    if out is None:
        out = torch.empty_like(q)
    _check(load().pkv_paged_attention_prefill(
        ctypes.byref(cache), _ptr(q), dtype_code(q.dtype), num_seqs, h, _ptr(cu_seqlens_q),
        total, int(max_q_len), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
        int(max_context_len), float(scale), _ptr(dev_err), _ptr(out), _stream(stream)),
        "pkv_paged_attention_prefill")
    return out


def pkv_swap_blocks(src, dst, block_pairs, dev_err=None, stream=None):
    """Move blocks src[l][pairs[i, 0]] -> dst[l][pairs[i, 1]] for every layer;
    `src` / `dst` are CacheDesc lists (device or pinned host pools)."""
    if isinstance(src, CacheDesc):
        src, dst = [src], [dst]
    if len(src) != len(dst):
        raise ValueError("src and dst need one descriptor per layer")
    a = (CacheDesc * len(src))(*src)
    b = (CacheDesc * len(dst))(*dst)
    _dense(block_pairs, "block_pairs")
    if block_pairs.dtype != torch.int64:
        raise ValueError("block_pairs must be int64 [n, 2]")
    _check(load().pkv_swap_blocks(a, b, len(src), _ptr(block_pairs), block_pairs.numel() // 2,
                                  _ptr(dev_err), _stream(stream)), "pkv_swap_blocks")


def pkv_testing_stream_copy(dst, src, stream=None):
    """Copy src into dst (same byte size) with SM loads and stores: the
    measurement reference for copies over a link (device <-> pinned host)."""
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("dst and src must have the same byte size")
    _check(load().pkv_testing_stream_copy(_ptr(dst), _ptr(src), nbytes, _stream(stream)),
           "pkv_testing_stream_copy")
    return dst


def pkv_block_hashes(token_ids, cu_seqlens, block_size, block_offsets=None, parent_hashes=None,
                     hashes=None, dev_err=None, stream=None):
    """Chained SHA-256 of every full block; returns uint8 [total_blocks, 32].
    `block_offsets` (int64 [num_seqs]) defaults to the running count of full
    blocks, which needs the lengths on the host (one device-to-host copy)."""
    _dense(token_ids, "token_ids")
    _dense(cu_seqlens, "cu_seqlens")
    if token_ids.dtype != torch.int32 or cu_seqlens.dtype != torch.int32:
        raise ValueError("token_ids and cu_seqlens must be int32")
    num_seqs = cu_seqlens.numel() - 1
    if block_offsets is None:
        full = torch.diff(cu_seqlens.to(torch.int64)) // block_size
        block_offsets = torch.cumsum(full, 0) - full
        total_blocks = int(full.sum().item())
    else:
        _dense(block_offsets, "block_offsets")
        total_blocks = hashes.shape[0] if hashes is not None else None
        if total_blocks is None:
            raise ValueError("pass `hashes` together with `block_offsets`")
    if hashes is None:
        hashes = torch.empty((max(total_blocks, 1), 32), dtype=torch.uint8,
                             device=token_ids.device)
    if parent_hashes is not None:
        _dense(parent_hashes, "parent_hashes")
    _check(load().pkv_block_hashes(_ptr(token_ids), _ptr(cu_seqlens), num_seqs,
                                   token_ids.numel(), int(block_size), _ptr(parent_hashes),
                                   _ptr(block_offsets), total_blocks, _ptr(hashes), _ptr(dev_err),
                                   _stream(stream)), "pkv_block_hashes")
    return hashes[:total_blocks]

