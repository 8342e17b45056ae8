"""CPU oracle for the paged KV-cache decode path (ctypes front of pkv_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  The
product library never imports, loads or calls it, and this package imports
nothing from the product.

Arrays cross this boundary as numpy arrays that hold the raw element bits:
``uint16`` for fp16 / bf16 data, ``uint8`` for E4M3 data.  Results come back in
float64.  Element type codes: 0 = fp16, 1 = bf16, 2 = FP8 E4M3.
"""
import ctypes
import os

import numpy as np

from . import build as _build

F16, BF16, E4M3 = 0, 1, 2

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        c_i64, c_i32, c_int = ctypes.c_int64, ctypes.c_int32, ctypes.c_int
        vp = ctypes.c_void_p
        lib.pkvo_dec_f16.argtypes = [ctypes.c_uint16]
        lib.pkvo_dec_f16.restype = ctypes.c_double
        lib.pkvo_dec_bf16.argtypes = [ctypes.c_uint16]
        lib.pkvo_dec_bf16.restype = ctypes.c_double
        lib.pkvo_dec_e4m3.argtypes = [ctypes.c_uint8]
        lib.pkvo_dec_e4m3.restype = ctypes.c_double
        lib.pkvo_enc_e4m3.argtypes = [ctypes.c_float]
        lib.pkvo_enc_e4m3.restype = ctypes.c_uint8
        lib.pkvo_dec_array.argtypes = [c_int, vp, c_i64, vp]
        lib.pkvo_dec_array.restype = None
        lib.pkvo_enc_e4m3_array.argtypes = [vp, c_i64, vp]
        lib.pkvo_enc_e4m3_array.restype = None
        lib.pkvo_kv_bytes_per_token.argtypes = [c_i64, c_i64, c_i64, c_i64]
        lib.pkvo_kv_bytes_per_token.restype = c_i64
        lib.pkvo_blocks_for_tokens.argtypes = [c_i64, c_i64]
        lib.pkvo_blocks_for_tokens.restype = c_i64
        lib.pkvo_gather.argtypes = [vp, c_int, c_i64, c_i32, c_i32, c_i32, vp, c_i32,
                                    c_i32, ctypes.c_double, vp]
        lib.pkvo_gather.restype = c_int
        lib.pkvo_kv_append.argtypes = [vp, vp, c_i64, c_i32, c_i32, c_i32, c_int,
                                       ctypes.c_float, ctypes.c_float, vp, vp, c_int,
                                       vp, c_i64]
        lib.pkvo_kv_append.restype = c_i64
        lib.pkvo_copy_blocks.argtypes = [vp, vp, c_i32, c_i64, c_i64, vp, c_i64]
        lib.pkvo_copy_blocks.restype = c_int
        lib.pkvo_paged_attention_decode.argtypes = [
            vp, vp, c_int, c_i64, c_i32, c_i32, c_i32, ctypes.c_float, ctypes.c_float,
            vp, c_int, c_i32, c_i32, vp, c_i32, vp, ctypes.c_float, vp, c_int]
        lib.pkvo_paged_attention_decode.restype = c_int
        lib.pkvo_attention_range.argtypes = [
            vp, vp, c_int, c_i64, c_i32, c_i32, c_i32, ctypes.c_float, ctypes.c_float,
            vp, c_int, c_i32, c_i32, vp, c_i32, vp, ctypes.c_float, c_i32, c_i32,
            vp, vp, vp, c_int]
        lib.pkvo_attention_range.restype = c_int
        _lib = lib
    return _lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def _contig(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != np.dtype(dtype):
        raise TypeError("expected %s, got %s" % (np.dtype(dtype), a.dtype))
    return a


def _check_rows(bt, cl, num_seqs):
    if bt.ndim != 2 or bt.shape[0] != num_seqs or cl.shape != (num_seqs,):
        raise ValueError("block_tables / context_lens do not match the number of sequences")


def _elem_np(code):
    return np.uint8 if code == E4M3 else np.uint16


# ---------------------------------------------------------------- elements

def decode(code, bits):
    """Exact value (float64) of every element of ``bits`` in format ``code``."""
    bits = _contig(bits, _elem_np(code))
    out = np.empty(bits.shape, np.float64)
    _load().pkvo_dec_array(code, _ptr(bits), bits.size, _ptr(out))
    return out


def encode_e4m3(y):
    """E4M3 code (round to nearest even, saturate to +-448) of fp32 values."""
    y = _contig(np.asarray(y, dtype=np.float32), np.float32)
    out = np.empty(y.shape, np.uint8)
    _load().pkvo_enc_e4m3_array(_ptr(y), y.size, _ptr(out))
    return out


# ---------------------------------------------------------------- sizing

def kv_bytes_per_token(num_kv_heads, head_dim, num_layers, elem_size):
    return int(_load().pkvo_kv_bytes_per_token(num_kv_heads, head_dim, num_layers, elem_size))


def blocks_for_tokens(n, block_size):
    return int(_load().pkvo_blocks_for_tokens(n, block_size))


# ---------------------------------------------------------------- cache ops

def gather(cache, cache_dtype, table_row, context_len, kv_head, scale=1.0):
    """Rows [context_len, head_dim] of one KV head in logical token order.

    ``cache`` has shape [num_blocks, num_kv_heads, block_size, head_dim]."""
    cache = _contig(cache, _elem_np(cache_dtype))
    nb, hkv, bs, d = cache.shape
    row = _contig(np.asarray(table_row, dtype=np.int32), np.int32)
    if row.ndim != 1 or row.size * bs < context_len:
        raise ValueError("the table row holds fewer blocks than the context needs")
    out = np.empty((context_len, d), np.float64)
    rc = _load().pkvo_gather(_ptr(cache), cache_dtype, nb, hkv, bs, d, _ptr(row),
                             context_len, kv_head, float(scale), _ptr(out))
    if rc != 0:
        raise IndexError("block table entry outside the pool")
    return out


def kv_append(k_cache, v_cache, cache_dtype, k, v, in_dtype, slot_mapping,
              k_scale=1.0, v_scale=1.0):
    """In-place append into numpy caches; returns the number of skipped
    out-of-pool slots.  ``k``/``v`` have shape [T, num_kv_heads, head_dim]."""
    for c in (k_cache, v_cache):
        if not c.flags.c_contiguous or c.dtype != np.dtype(_elem_np(cache_dtype)):
            raise TypeError("cache must be a C-contiguous array of the cache element type")
    nb, hkv, bs, d = k_cache.shape
    k = _contig(k, _elem_np(in_dtype))
    v = _contig(v, _elem_np(in_dtype))
    slots = _contig(np.asarray(slot_mapping, dtype=np.int64), np.int64)
    n = _load().pkvo_kv_append(_ptr(k_cache), _ptr(v_cache), nb, hkv, bs, d, cache_dtype,
                               float(k_scale), float(v_scale), _ptr(k), _ptr(v), in_dtype,
                               _ptr(slots), slots.size)
    if n < 0:
        raise ValueError("unsupported dtype pairing")
    return int(n)


def copy_blocks(k_caches, v_caches, pairs):
    """In-place copy of whole blocks for every layer; ``pairs`` is [n, 2]."""
    layers = len(k_caches)
    nb = k_caches[0].shape[0]
    block_bytes = k_caches[0][0].nbytes
    for c in list(k_caches) + list(v_caches):
        if not c.flags.c_contiguous or c.shape[0] != nb or c[0].nbytes != block_bytes:
            raise TypeError("caches must be C-contiguous and alike")
    kp = (ctypes.c_void_p * layers)(*[c.ctypes.data for c in k_caches])
    vp = (ctypes.c_void_p * layers)(*[c.ctypes.data for c in v_caches])
    pairs = _contig(np.asarray(pairs, dtype=np.int64).reshape(-1, 2), np.int64)
    rc = _load().pkvo_copy_blocks(kp, vp, layers, nb, block_bytes, _ptr(pairs), pairs.shape[0])
    if rc != 0:
        raise IndexError("copy pair outside the pool")


def paged_attention_decode(k_cache, v_cache, cache_dtype, q, q_dtype, block_tables,
                           context_lens, scale, k_scale=1.0, v_scale=1.0, nthreads=0):
    """Exact decode attention; returns float64 [num_seqs, num_heads, head_dim]."""
    k_cache = _contig(k_cache, _elem_np(cache_dtype))
    v_cache = _contig(v_cache, _elem_np(cache_dtype))
    nb, hkv, bs, d = k_cache.shape
    q = _contig(q, _elem_np(q_dtype))
    s, h, dq = q.shape
    assert dq == d
    bt = _contig(np.asarray(block_tables, dtype=np.int32), np.int32)
    cl = _contig(np.asarray(context_lens, dtype=np.int32), np.int32)
    _check_rows(bt, cl, s)
    out = np.zeros((s, h, d), np.float64)
    rc = _load().pkvo_paged_attention_decode(
        _ptr(k_cache), _ptr(v_cache), cache_dtype, nb, hkv, bs, d,
        float(k_scale), float(v_scale), _ptr(q), q_dtype, s, h, _ptr(bt), bt.shape[1],
        _ptr(cl), float(np.float32(scale)), _ptr(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle decode failed (%d)" % rc)
    return out


def attention_range(k_cache, v_cache, cache_dtype, q, q_dtype, block_tables, context_lens,
                    scale, t_begin, t_end, k_scale=1.0, v_scale=1.0, nthreads=0):
    """Unnormalised attention over tokens [t_begin, t_end) of each context.

    Returns (o, m, l): o = sum_t exp(x_t - m) v_t [S, H, D], m = max logit,
    l = sum_t exp(x_t - m)."""
    k_cache = _contig(k_cache, _elem_np(cache_dtype))
    v_cache = _contig(v_cache, _elem_np(cache_dtype))
    nb, hkv, bs, d = k_cache.shape
    q = _contig(q, _elem_np(q_dtype))
    s, h, _ = q.shape
    bt = _contig(np.asarray(block_tables, dtype=np.int32), np.int32)
    cl = _contig(np.asarray(context_lens, dtype=np.int32), np.int32)
    _check_rows(bt, cl, s)
    o = np.zeros((s, h, d), np.float64)
    m = np.zeros((s, h), np.float64)
    l = np.zeros((s, h), np.float64)
    rc = _load().pkvo_attention_range(
        _ptr(k_cache), _ptr(v_cache), cache_dtype, nb, hkv, bs, d,
        float(k_scale), float(v_scale), _ptr(q), q_dtype, s, h, _ptr(bt), bt.shape[1],
        _ptr(cl), float(np.float32(scale)), int(t_begin), int(t_end),
        _ptr(o), _ptr(m), _ptr(l), int(nthreads))
    if rc != 0:
        raise ValueError("oracle range attention failed (%d)" % rc)
    return o, m, l


def paged_attention_prefill(k_cache, v_cache, cache_dtype, q, q_dtype, cu_seqlens_q,
                            block_tables, context_lens, scale, k_scale=1.0, v_scale=1.0,
                            nthreads=0):
    """Exact causal prefill attention over the paged cache; float64 [total_q, H, D].

    Sequence s brings n_s = cu_seqlens_q[s+1] - cu_seqlens_q[s] new tokens
    whose K/V are already in the cache as the last n_s of its context_lens[s]
    tokens (the prompt's K/V are all computed and stored in one pass:
    「KV Cache从原理到实战」 §2.3).  Query j of sequence s sits at position
    p = context_lens[s] - n_s + j and, like the decode token, attends to
    itself and every earlier token (「KV 缓存与分页注意力」 §02): its output is
    the decode attention of one query over a context of p + 1 tokens.  The
    oracle therefore expands every query row into one decode row with its
    sequence's block table and context length p + 1."""
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    cl = np.asarray(context_lens, dtype=np.int64)
    bt = np.asarray(block_tables, dtype=np.int32)
    num_seqs = len(cl)
    if cu.shape != (num_seqs + 1,) or cu[0] != 0 or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens_q must be ascending from 0 with num_seqs + 1 entries")
    n = np.diff(cu)
    if np.any(n > cl):
        raise ValueError("a sequence has more new tokens than context")
    total = int(cu[-1])
    if q.shape[0] != total:
        raise ValueError("q must hold cu_seqlens_q[-1] rows")
    seq_of_row = np.repeat(np.arange(num_seqs), n)
    j = np.arange(total) - cu[seq_of_row]
    pos = cl[seq_of_row] - n[seq_of_row] + j
    rows_bt = bt[seq_of_row] if total else np.zeros((0, bt.shape[1]), np.int32)
    return paged_attention_decode(k_cache, v_cache, cache_dtype, q, q_dtype, rows_bt,
                                  (pos + 1).astype(np.int32), scale, k_scale, v_scale,
                                  nthreads)


def swap_blocks(src_k, src_v, dst_k, dst_v, pairs):
    """Block swap between two pools (device cache <-> host memory), in place.

    When blocks run short, all of a sequence's blocks move to CPU memory and
    come back when the sequence runs again (「KV 缓存与分页注意力」 §09).  For each
    (src, dst) pair and every layer l: dst_k[l][dst] = src_k[l][src] and the
    same for V, byte for byte.  The two pools are different arrays, so the
    order of the pairs does not matter unless two pairs name the same dst (a
    caller error; the later pair wins here).  Raises IndexError when a pair
    lies outside its pool."""
    pairs = np.asarray(pairs, dtype=np.int64).reshape(-1, 2)
    for l in range(len(src_k)):
        ns, nd = src_k[l].shape[0], dst_k[l].shape[0]
        for src, dst in pairs:
            if not (0 <= src < ns and 0 <= dst < nd):
                raise IndexError("swap pair outside its pool")
            dst_k[l][dst] = src_k[l][src]
            dst_v[l][dst] = src_v[l][src]


def block_hashes(token_ids, cu_seqlens, block_size, parent_hashes=None):
    """Content hashes of every full block, chained over the blocks before it.

    Prefix caching gives each full block a hash of its tokens and of all the
    content in front of it, so that equal prompt openings map to the same
    blocks (「KV 缓存与分页注意力」 §11; 「KV Cache从原理到实战」 §4.2).  Here
    h_i = SHA-256(h_{i-1} || tokens of block i as little-endian int32), with
    h_{-1} = parent_hashes[s] (32 zero bytes when absent); a partial last block
    has no hash.  Returns a list, per sequence, of 32-byte digests."""
    import hashlib
    toks = np.asarray(token_ids, dtype=np.int32)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    out = []
    for s in range(len(cu) - 1):
        seq = toks[cu[s]:cu[s + 1]]
        h = bytes(32) if parent_hashes is None else bytes(np.asarray(parent_hashes[s],
                                                                     np.uint8))
        hs = []
        for b in range(len(seq) // block_size):
            msg = h + seq[b * block_size:(b + 1) * block_size].astype("<i4").tobytes()
            h = hashlib.sha256(msg).digest()
            hs.append(h)
        out.append(hs)
    return out
