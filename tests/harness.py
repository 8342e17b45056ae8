"""Shared test plumbing: one workload driven through the CUDA library and
through the oracle, step by step, from the same seeded inputs.

Both sides start from caches filled with 0xFF bytes (a NaN in every element
type), so that any read of an unwritten slot shows up in the results.
"""
import os

import numpy as np
import torch

import oracle
from paged_kv_cache_130_gb300 import binding as B
from paged_kv_cache_130_gb300 import workloads as W

SENTINEL = 0xFF
TORCH_DT = {W.F16: torch.float16, W.BF16: torch.bfloat16, W.E4M3: torch.uint8}
ATOL = 2e-3
RTOL = 2e-3


def build_library():
    from paged_kv_cache_130_gb300 import build as pkv_build
    pkv_build.build()
    return B.load()


def to_device(bits, code, device="cuda"):
    """uint16 / uint8 numpy bits -> torch tensor of the element type."""
    a = np.ascontiguousarray(bits)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(TORCH_DT[code])
    else:
        t = torch.from_numpy(a)
    return t.to(device)


def to_bits(t):
    """Device tensor -> numpy bits (uint16 for 16-bit types, uint8 for bytes)."""
    t = t.detach().contiguous().cpu()
    if t.element_size() == 2:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.uint8).numpy()


class GpuRun:
    """A workload's cache and inputs on the device, driven through the C ABI."""

    def __init__(self, w, device="cuda"):
        self.w = w
        self.device = device
        shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
        cdt = TORCH_DT[w.cache_dtype]
        nbytes = int(np.prod(shape)) * (1 if w.cache_dtype == W.E4M3 else 2)
        self.k_cache = torch.full((nbytes,), SENTINEL, dtype=torch.uint8, device=device).view(cdt)
        self.v_cache = torch.full((nbytes,), SENTINEL, dtype=torch.uint8, device=device).view(cdt)
        self.k_cache = self.k_cache.view(shape)
        self.v_cache = self.v_cache.view(shape)
        self.desc = B.cache_desc(self.k_cache, self.v_cache, w.k_scale, w.v_scale)
        self.q = to_device(w.q, w.io_dtype, device)
        self.block_tables = torch.from_numpy(w.block_tables).to(device)
        self.context_lens = torch.from_numpy(w.context_lens).to(device)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=device)

    def append(self, slots, k_bits, v_bits):
        k = to_device(k_bits, self.w.io_dtype, self.device)
        v = to_device(v_bits, self.w.io_dtype, self.device)
        s = torch.from_numpy(np.ascontiguousarray(slots)).to(self.device)
        B.pkv_kv_append(self.desc, k, v, s, dev_err=self.dev_err)

    def prefill(self):
        for slots, k, v in self.w.prefill():
            self.append(slots, k, v)

    def copy(self):
        if len(self.w.copy_pairs):
            pairs = torch.from_numpy(self.w.copy_pairs).to(self.device)
            B.pkv_copy_blocks(self.desc, pairs, dev_err=self.dev_err)

    def step(self):
        k, v = self.w.step_values()
        self.append(self.w.step_slots, k, v)

    def decode(self, partition_size=None):
        ps = self.w.partition_size if partition_size is None else partition_size
        return B.pkv_paged_attention_decode(self.desc, self.q, self.block_tables,
                                            self.context_lens, self.w.max_context_len,
                                            self.w.scale, partition_size=ps,
                                            dev_err=self.dev_err)

    def decode_shared(self, partition_size=None, groups=None, max_group_size=None,
                      max_prefix_blocks=None):
        """Decode through the shared-prefix entry point; groups default to the
        batch's own (Workload.prefix_groups)."""
        w = self.w
        ps = w.partition_size if partition_size is None else partition_size
        begin, blocks = w.prefix_groups() if groups is None else groups
        sizes = np.diff(begin)
        mgs = int(sizes.max()) if max_group_size is None else max_group_size
        mpb = int(blocks.max()) if max_prefix_blocks is None else max_prefix_blocks
        return B.pkv_paged_attention_decode_shared_prefix(
            self.desc, self.q, self.block_tables, self.context_lens, w.max_context_len,
            torch.from_numpy(np.ascontiguousarray(begin, np.int32)).to(self.device),
            torch.from_numpy(np.ascontiguousarray(blocks, np.int32)).to(self.device),
            mgs, mpb, w.scale, partition_size=ps, dev_err=self.dev_err)

    def prefill_attention(self):
        """Causal prefill of the workload's new tokens (after step())."""
        w = self.w
        cu = torch.from_numpy(w.cu_seqlens_q).to(self.device)
        return B.pkv_paged_attention_prefill(self.desc, self.q, cu, w.max_q_len,
                                             self.block_tables, self.context_lens,
                                             w.max_context_len, w.scale, dev_err=self.dev_err)

    def run_all(self, partition_size=None):
        self.prefill()
        self.copy()
        self.step()
        out = self.decode(partition_size)
        torch.cuda.synchronize()
        return out


class OracleRun:
    """The same workload on host caches through the oracle."""

    def __init__(self, w, sequences=None):
        self.w = w
        shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
        dt = np.uint8 if w.cache_dtype == W.E4M3 else np.uint16
        self.k_cache = np.empty(shape, dt)
        self.v_cache = np.empty(shape, dt)
        self.k_cache.view(np.uint8)[...] = SENTINEL
        self.v_cache.view(np.uint8)[...] = SENTINEL
        self.sequences = sequences

    def append(self, slots, k, v):
        return oracle.kv_append(self.k_cache, self.v_cache, self.w.cache_dtype, k, v,
                                self.w.io_dtype, slots, self.w.k_scale, self.w.v_scale)

    def prefill(self):
        for slots, k, v in self.w.prefill():
            self.append(slots, k, v)

    def copy(self):
        if len(self.w.copy_pairs):
            oracle.copy_blocks([self.k_cache], [self.v_cache], self.w.copy_pairs)

    def step(self):
        k, v = self.w.step_values()
        self.append(self.w.step_slots, k, v)

    def decode(self, seqs=None):
        w = self.w
        q, bt, cl = w.q, w.block_tables, w.context_lens
        if seqs is not None:
            q, bt, cl = q[seqs], bt[seqs], cl[seqs]
        return oracle.paged_attention_decode(self.k_cache, self.v_cache, w.cache_dtype, q,
                                             w.io_dtype, bt, cl, w.scale, w.k_scale, w.v_scale)

    def prefill_attention(self, rows=None):
        """Oracle prefill of the new tokens; `rows` picks query rows (each is
        the decode of its position's causal context)."""
        w = self.w
        if rows is None:
            return oracle.paged_attention_prefill(
                self.k_cache, self.v_cache, w.cache_dtype, w.q, w.io_dtype, w.cu_seqlens_q,
                w.block_tables, w.context_lens, w.scale, w.k_scale, w.v_scale)
        cu = w.cu_seqlens_q.astype(np.int64)
        rows = np.asarray(rows, dtype=np.int64)
        seq = np.searchsorted(cu, rows, side="right") - 1
        n = cu[seq + 1] - cu[seq]
        pos = w.context_lens[seq].astype(np.int64) - n + (rows - cu[seq])
        return oracle.paged_attention_decode(
            self.k_cache, self.v_cache, w.cache_dtype, w.q[rows], w.io_dtype,
            w.block_tables[seq], (pos + 1).astype(np.int32), w.scale, w.k_scale, w.v_scale)

    def run_all(self):
        self.prefill()
        self.copy()
        self.step()
        return self.decode()


def out_to_double(out):
    return out.detach().float().cpu().numpy().astype(np.float64)


def half_ulp(ref, out_dtype):
    """Half the spacing of the output format (fp16 / bf16) at |ref|: the most
    that the one final round-to-nearest of the output can move a value."""
    a = np.abs(np.asarray(ref, np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    if out_dtype == W.BF16:
        e = np.maximum(e, -126.0)
        return np.ldexp(1.0, (e - 8).astype(np.int64))
    e = np.maximum(e, -14.0)
    return np.ldexp(1.0, (e - 11).astype(np.int64))


def assert_attention_close(got, ref, what="", out_dtype=W.F16):
    """|got - ref| <= 2e-3 + 2e-3 |ref| elementwise.

    For bf16 outputs the bound also allows half an ulp of bf16 at |ref|: the
    kernel's fp32 result is rounded once to bf16, and that rounding alone can
    move a value by up to 2^-8 |ref|, more than 2e-3 |ref|.  For fp16 outputs
    half an ulp is at most 2^-11 |ref|, which the plain bound already covers,
    so fp16 outputs are held to the plain bound.  Returns the worst
    err / bound ratio (also recorded in WORST_RATIO under `what`)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite output" % what
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    if out_dtype == W.BF16:
        bound = bound + half_ulp(ref, out_dtype)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError("%s: %d of %d outside tolerance; worst at %s: got %r ref %r"
                             % (what, int(bad.sum()), bad.size, i, got[i], ref[i]))
    ratio = float((err / bound).max()) if err.size else 0.0
    key = "%s (%s)" % (what, "bf16" if out_dtype == W.BF16 else "fp16")
    WORST_RATIO[key] = max(ratio, WORST_RATIO.get(key, 0.0))
    return ratio


# worst err / bound ratio seen per check name during the session
WORST_RATIO = {}


def gpu_available():
    return torch.cuda.is_available()


def oracle_threads():
    return int(os.environ.get("PKV_ORACLE_THREADS", "0"))


def segment_sequences(w, seg):
    """Sequences whose tokens a prefill segment holds."""
    return w.segment_sequences(seg)


def prefill_both(w, g, o, only=None, threads=8):
    """Prefill the GPU cache with every segment and the oracle's cache with the
    segments of `only` (all when None); values are drawn once, in parallel."""
    import concurrent.futures as cf
    segs = list(w.segments)
    with cf.ThreadPoolExecutor(threads) as ex:
        futs = [ex.submit(w.values, seg.key, len(seg.slots)) for seg in segs[:threads * 2]]
        for i, seg in enumerate(segs):
            k, v = futs[i].result()
            futs[i] = None
            j = i + threads * 2
            if j < len(segs):
                futs.append(ex.submit(w.values, segs[j].key, len(segs[j].slots)))
            g.append(seg.slots, k, v)
            if o is not None and (only is None or segment_sequences(w, seg) & set(only)):
                o.append(seg.slots, k, v)
