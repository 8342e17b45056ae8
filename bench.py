"""Benchmark of the paged decode step on GB300.

One step = the whole hot path over one batch: the copy-on-write block copies
(when the workload has any), the append of the step's new tokens, and decode
attention over every sequence (partition kernel + log-sum-exp reduce).  The
cache is pre-filled once (untimed).  The step is captured as one CUDA graph
with event nodes between its stages, and ``value`` is the decode call's
interval inside it (``separate_graphs`` keeps the same with the step as two
graphs, events between their replays); the roofline's kernel is launched
back to back, and once more each launch alone after an L2 read.  The decode
inputs of every benchmark layer exceed the 129 MB L2, so no flush is needed
(``--flush write`` adds a 512 MiB write between steps, ``--flush read`` a
512 MiB read, which leaves L2 holding clean lines of another buffer).

Output: one JSON line on rank 0.  ``value`` is decode KV-read GB/s: algorithmic
bytes of one decode (every cached K/V element once per KV head -- a block that
forked sequences share is counted once when the shared-prefix call reads it
once --, q, out, the used block-table entries and the context lengths) over the
decode time measured with CUDA events on the launch stream, summed over all
ranks' work and divided by the slowest rank's time (replicas: every rank
decodes its own batch).  The default run (OPT-13B layer) also times the GQA,
copy-on-write and long E4M3 layers the same way, under ``configs``.

``--impl reference`` times the CPU oracle on the host cores on a bounded sample
of the same workload instead (rank 0 only).
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode-attention KV-read GB/s (fraction of HBM peak); decode tokens/s"
DEFAULT_WORKLOAD = "opt13b_f16"
MODEL_LAYERS = {"opt13b_f16": 40, "llama2_70b_bf16_gqa": 80, "llama2_7b_fp8_long": 32,
                "cow_parallel_sampling_f16": 40, "tiny_f16": 1}
FLUSH_BYTES = 512 << 20
FALLBACK_HBM_GBS = 6800.0
# DRAM bytes (read + write) per launch of the timed kernel from a one-pass ncu
# capture (dram__bytes_read.sum, dram__bytes_write.sum, gpu__time_duration.sum)
# of the full-size workload, valid while the sources hash to "src_sha" (else
# reported as null); "profile" names the summary under profiles/ that prints
# the figures and the command.
NCU_TRAFFIC = {
    "opt13b_f16": {"bytes_per_launch": 366086656 + 2871296, "src_sha": "a2cc1717bfee0912",
                   "profile": "profiles/decode_stream_kernel_opt13b_f16.md"},
    "llama2_70b_bf16_gqa": {"bytes_per_launch": 642888960 + 3087872,
                            "src_sha": "a2cc1717bfee0912",
                            "profile": "profiles/decode_mma_kernel_llama2_70b_bf16_gqa.md"},
    "llama2_7b_fp8_long": {"bytes_per_launch": 2497219328 + 6611456,
                           "src_sha": "a2cc1717bfee0912",
                           "profile": "profiles/decode_stream_kernel_llama2_7b_fp8_long.md"},
    # the single-pass shared-prefix kernel (the whole decode call)
    "cow_parallel_sampling_f16:shared-prefix": {
        "bytes_per_launch": 381789696 + 3032832, "src_sha": "a2cc1717bfee0912",
        "profile": "profiles/decode_group_kernel_cow_parallel_sampling_f16.md"},
}
DECODE_SOURCES = ("decode.cu", "decode_stream.cu", "decode_group.cu", "decode_common.cuh",
                  "pkv_common.cuh", "tc_common.cuh", "pkv_api.cu")
# the same for the prefill kernel
NCU_PREFILL_TRAFFIC = {
    "prefill_llama2_7b_bf16": {"bytes_per_launch": 645102080 + 61541120,
                               "src_sha": "6c93987b8c1a6914",
                               "profile": "profiles/prefill_ws_kernel_prefill_llama2_7b_bf16.md"},
    "prefill_llama2_70b_gqa_chunked_bf16": {
        "bytes_per_launch": 177549824 + 23233280, "src_sha": "6c93987b8c1a6914",
        "profile": "profiles/prefill_ws_kernel_prefill_llama2_7b_bf16.md"},
}
# the same for the block-hash kernel
NCU_HASH_TRAFFIC = {
    "hash_prompts": {"bytes_per_launch": 21091328 + 0, "src_sha": "9fc632474980a784",
                     "profile": "profiles/block_hash_kernel_hash_prompts.md"},
}
HASH_SOURCES = ("block_hash.cu", "pkv_common.cuh")
PREFILL_SOURCES = ("prefill_ws.cu", "tc_common.cuh", "pkv_common.cuh")


def percentiles(ms):
    """p10 / median / p90 of per-step times (ms), nearest rank."""
    v = sorted(ms)
    if not v:
        return None
    pick = lambda q: v[min(len(v) - 1, max(0, int(round(q * (len(v) - 1)))))]
    return {"p10": pick(0.1), "p50": pick(0.5), "p90": pick(0.9)}


def src_sha(names):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "paged_kv_cache_130_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def decode_src_sha():
    return src_sha(DECODE_SOURCES)


def shares_prefixes(w):
    """Whether the shared-prefix kernel takes this workload's shape."""
    from paged_kv_cache_130_gb300 import workloads as W
    group = w.num_heads // w.num_kv_heads
    return (w.cache_dtype == w.io_dtype and w.cache_dtype != W.E4M3 and 1 <= group <= 16
            and w.block_size in (16, 32) and w.head_dim in (64, 128))


def shared_single_pass(w, max_group, sms):
    """Whether the library decodes this batch's shared prefixes in a single
    pass: partition size left to the library, contexts of at most 4096
    tokens, and at least one (group, KV head, row tile) CTA per SM."""
    group = w.num_heads // w.num_kv_heads
    rows = max_group * group
    rt = 16 if rows > 8 else 8
    _, blocks = w.prefix_groups()
    ctas = len(blocks) * (-(-rows // rt)) * w.num_kv_heads
    return w.partition_size == 0 and w.max_context_len <= 4096 and ctas >= sms


def decode_kernel_name(w):
    """Which partition kernel the library runs for this workload: grouped
    16-bit heads go to the tensor-core kernel, everything else streams."""
    from paged_kv_cache_130_gb300 import workloads as W
    group = w.num_heads // w.num_kv_heads
    grouped = (2 <= group <= 16 and w.cache_dtype == w.io_dtype and w.cache_dtype != W.E4M3
               and w.block_size % 16 == 0)
    return "decode_mma_kernel" if grouped else "decode_stream_kernel"


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-graphs", action="store_true")
    ap.add_argument("--shared-prefix", default="auto", choices=["auto", "off"],
                    help="auto: decode batches with forked sequences through the "
                         "shared-prefix entry point (each shared block read once per group)")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="a smaller batch of the same decode workload (profiler "
                         "captures); the line's config names the batch")
    ap.add_argument("--configs", default="auto",
                    help="auto: the default run also times the other decode workloads "
                         "(GQA, copy-on-write parallel sampling, long E4M3) under a "
                         "`configs` key; none: the headline workload only; or a "
                         "comma-separated list of workload names")
    ap.add_argument("--flush", default="none", choices=["none", "write", "read"],
                    help="none: the decode inputs alone exceed L2; write: also write "
                         "512 MiB between steps")
    return ap.parse_args(argv)


# ------------------------------------------------------------------ ranks

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def slowest(seconds, device=None):
    """Each timing maximised over the ranks of the default process group
    (unchanged when there is no group).  `device` is where the reduction
    tensor lives: the rank's GPU under NCCL, the CPU under gloo."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(x) for x in seconds]
    t = torch.tensor([float(x) for x in seconds], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def whole_job_rate(units_per_rank, seconds_slowest, world):
    """Replicas: every rank processes the same units; the job rate is all the
    ranks' units over the slowest rank's time."""
    return units_per_rank * world / seconds_slowest if seconds_slowest > 0 else 0.0


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed loop runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names[1:], parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ peaks

def tensor_peak():
    """Measured dense bf16 TFLOP/s (burst: the kernel is timed alone); fp16 runs
    at the same nominal rate on this part."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ oracle timing

def oracle_decode_sample(w, state, seqs, reps):
    """Time the oracle's decode on `seqs` of the workload, `reps` times."""
    import oracle
    q, bt, cl = w.q[seqs], w.block_tables[seqs], w.context_lens[seqs]
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.paged_attention_decode(state.k_cache, state.v_cache, w.cache_dtype, q, w.io_dtype,
                                      bt, cl, w.scale, w.k_scale, w.v_scale)
    return time.perf_counter() - t0


def sample_bytes(w, seqs):
    ctx = w.context_lens[seqs].astype(np.int64)
    kv = int(ctx.sum()) * w.num_kv_heads * w.head_dim * 2 * w.cache_elem_bytes
    qo = 2 * len(seqs) * w.num_heads * w.head_dim * 2
    bt = 4 * int(((ctx + w.block_size - 1) // w.block_size).sum())
    return kv + qo + bt + 4 * len(seqs)


class HostState:
    """Host caches written through the oracle (the CPU arm's inputs).

    `prefill`: the workload's (slots, k, v) batches, or None to draw the
    segments here; `seqs`: only the segments these sequences read (all when
    None).  The copy-on-write pairs and the step's tokens are always applied."""

    def __init__(self, w, prefill=None, seqs=None, threads=8):
        import oracle
        shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
        dt = np.uint8 if w.cache_elem_bytes == 1 else np.uint16
        self.k_cache = np.zeros(shape, dt)
        self.v_cache = np.zeros(shape, dt)
        if prefill is None:
            segs = w.segments if seqs is None else w.segments_of(seqs)
            prefill = w.prefill(threads=threads, segments=segs)
        for slots, k, v in prefill:
            oracle.kv_append(self.k_cache, self.v_cache, w.cache_dtype, k, v, w.io_dtype, slots,
                             w.k_scale, w.v_scale)
        if len(w.copy_pairs):
            oracle.copy_blocks([self.k_cache], [self.v_cache], w.copy_pairs)
        k, v = w.step_values()
        oracle.kv_append(self.k_cache, self.v_cache, w.cache_dtype, k, v, w.io_dtype,
                         w.step_slots, w.k_scale, w.v_scale)


def sample_sequences(w, cap_bytes):
    """Leading sequences whose K/V fit `cap_bytes` (at least one): the part
    of a workload the host prepares for a bounded oracle run."""
    per = (w.context_lens.astype(np.int64) * w.num_kv_heads * w.head_dim * 2
           * w.cache_elem_bytes)
    n = int(np.searchsorted(np.cumsum(per), cap_bytes, side="right"))
    return np.arange(max(1, min(w.num_seqs, n)))


def pick_sample(w, budget_s, host_state, seqs=None):
    """Sequences (out of `seqs`, default all) and repetitions for a bounded
    oracle run (~budget_s seconds)."""
    seqs = np.arange(w.num_seqs) if seqs is None else np.asarray(seqs)
    one = oracle_decode_sample(w, host_state, seqs[:1], 1)
    per_seq = max(one, 1e-4)
    n = int(min(len(seqs), max(1, budget_s / per_seq)))
    seqs = seqs[:n]
    reps = 1
    t = oracle_decode_sample(w, host_state, seqs, 1)
    if t < budget_s / 4:
        reps = int(max(1, min(20, budget_s / max(t, 1e-4))))
    return seqs, reps


def run_reference(args, w, prefill=None):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    hs = HostState(w, prefill)
    cores = os.cpu_count() or 1
    seqs, _ = pick_sample(w, 20.0 / max(1, args.steps + args.warmup), hs)
    for _ in range(args.warmup):
        oracle_decode_sample(w, hs, seqs, 1)
    t = oracle_decode_sample(w, hs, seqs, args.steps)
    per = t / max(1, args.steps)
    gbs = sample_bytes(w, seqs) / per / 1e9
    line = {"metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": workload_config(w),
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": "decode of %d of %d sequences per step (%d context "
                                       "tokens)" % (len(seqs), w.num_seqs,
                                                    int(w.context_lens[seqs].sum()))},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    return line


# ------------------------------------------------------------------ GPU arm

def workload_config(w):
    return {"workload": w.name, "num_seqs": w.num_seqs, "num_heads": w.num_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "block_size": w.block_size, "num_blocks": w.num_blocks,
            "cache_dtype": {0: "f16", 1: "bf16", 2: "e4m3"}[w.cache_dtype],
            "q_dtype": {0: "f16", 1: "bf16"}[w.io_dtype],
            "context_tokens": int(w.context_lens.sum()),
            "max_context_len": w.max_context_len,
            "copy_pairs": int(len(w.copy_pairs)),
            "step_tokens": int(len(w.step_slots)),
            "l2": "decode inputs (%.0f MB of K/V per step) exceed the 129 MB L2; no flush"
                  % (w.kv_bytes() / 1e6),
            "parallelism": "replicas"}


def step_graph(stream, stages):
    """The stages of one step captured into ONE CUDA graph, with an event node
    before the first stage and after each, so that each stage is timed inside
    the step as an engine that captures its whole step runs it (no graph
    launch between stages).  Returns a function that replays the graph, waits
    for it and returns each stage's milliseconds; None where this PyTorch
    cannot record timing events inside a capture."""
    import torch
    try:
        evs = [torch.cuda.Event(enable_timing=True, external=True)
               for _ in range(len(stages) + 1)]
    except TypeError:
        return None
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        evs[0].record()
        for i, fn in enumerate(stages):
            fn()
            evs[i + 1].record()

    def run():
        g.replay()
        evs[-1].synchronize()
        return [evs[i].elapsed_time(evs[i + 1]) for i in range(len(stages))]
    return run


def run_gpu(args, w, cpu_budget_s=15.0, sample_cap_bytes=None, threads=8):
    """Time the decode step of workload `w` on this rank's GPU; returns the
    JSON line (rank 0) or None.  The cache is filled from the workload's
    seeded values, drawn in a thread pool; the oracle's CPU baseline runs on
    the sequences whose K/V fit `sample_cap_bytes` (all when None)."""
    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from paged_kv_cache_130_gb300 import binding as B
    from paged_kv_cache_130_gb300 import build as pkv_build
    pkv_build.build()
    B.load()

    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)

    shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    cdt = {0: torch.float16, 1: torch.bfloat16, 2: torch.uint8}[w.cache_dtype]
    iodt = {0: torch.float16, 1: torch.bfloat16}[w.io_dtype]
    k_cache = torch.zeros(shape, dtype=cdt, device=dev)
    v_cache = torch.zeros(shape, dtype=cdt, device=dev)
    desc = B.cache_desc(k_cache, v_cache, w.k_scale, w.v_scale)

    def dev16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(iodt).to(dev)

    for slots, k, v in w.prefill(threads=threads):
        B.pkv_kv_append(desc, dev16(k), dev16(v), torch.from_numpy(slots).to(dev))
    q = dev16(w.q)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    sk, sv = w.step_values()
    step_k, step_v = dev16(sk), dev16(sv)
    step_slots = torch.from_numpy(w.step_slots).to(dev)
    pairs = torch.from_numpy(w.copy_pairs).to(dev) if len(w.copy_pairs) else None
    ps = B.pkv_decode_partition_size(desc, w.num_seqs, w.num_heads, w.max_context_len,
                                     w.partition_size)
    grp_begin, grp_blocks = w.prefix_groups()
    shared = (args.shared_prefix == "auto" and int(grp_blocks.max(initial=0)) > 0
              and shares_prefixes(w))
    single = False
    if shared:
        gb = torch.from_numpy(grp_begin).to(dev)
        gp = torch.from_numpy(grp_blocks).to(dev)
        max_group = int(np.diff(grp_begin).max())
        max_prefix = int(grp_blocks.max())
        ws_bytes = B.pkv_shared_prefix_workspace_bytes(desc, w.num_seqs, w.num_heads,
                                                       w.max_context_len, ps)
        # the library's route for this call (the workload leaves the split to
        # the library, partition size 0): the single pass when its CTAs cover
        # the GPU, as pkv_testing_set_shared_prefix_path documents
        single = shared_single_pass(w, max_group, torch.cuda.get_device_properties(dev)
                                    .multi_processor_count)
        # the split route's partition size, as the library resolves it
        shared_ps = w.partition_size
    else:
        ws_bytes = B.pkv_decode_workspace_bytes(desc, w.num_seqs, w.num_heads,
                                                w.max_context_len, ps)
    workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    flush = torch.empty(FLUSH_BYTES if args.flush != "none" else 16, dtype=torch.uint8,
                        device=dev)
    maxp = -(-w.max_context_len // ps)
    launches_per_step = 1 + (1 if pairs is not None else 0) + 1 + (1 if maxp > 1 else 0)
    if shared:
        launches_per_step = 1 + (1 if pairs is not None else 0) + (1 if single else 3)

    def pre():
        if pairs is not None:
            B.pkv_copy_blocks(desc, pairs)
        B.pkv_kv_append(desc, step_k, step_v, step_slots)

    def decode():
        if shared:
            B.pkv_paged_attention_decode_shared_prefix(
                desc, q, bt, cl, w.max_context_len, gb, gp, max_group, max_prefix, w.scale,
                partition_size=shared_ps, workspace=workspace, out=out)
        else:
            B.pkv_paged_attention_decode(desc, q, bt, cl, w.max_context_len, w.scale,
                                         partition_size=ps, workspace=workspace, out=out)

    def partitions():
        # with shared prefixes the prefix and partition kernels split the
        # reads between them: the roofline takes the whole decode call
        if shared:
            decode()
        else:
            B.pkv_paged_attention_partitions(desc, q, bt, cl, w.max_context_len, w.scale,
                                             partition_size=ps, workspace=workspace, out=out)

    flush_sink = torch.zeros(1, dtype=torch.int64, device=dev)

    def maybe_flush(i):
        if args.flush == "write":
            flush.fill_(i & 0xff)
        elif args.flush == "read":
            flush_sink.add_(flush.view(torch.int64).sum())

    torch.cuda.synchronize()
    for i in range(args.warmup):
        maybe_flush(i)
        pre()
        decode()
        partitions()
    torch.cuda.synchronize()

    # Each stage is captured once as a CUDA graph and replayed: a replay costs
    # the host a few microseconds, so the GPU never waits for Python between
    # the events that bracket a stage.
    stages = {"pre": pre, "decode": decode, "partitions": partitions}
    replay = dict(stages)
    if not args.no_graphs:
        for name, fn in stages.items():
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            replay[name] = g.replay
        torch.cuda.synchronize()

    clocks = ClockSampler(local) if not args.no_clocks else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    evs = []
    for i in range(args.steps):
        maybe_flush(i)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e2 = torch.cuda.Event(enable_timing=True)
        e0.record()
        replay["pre"]()
        e1.record()
        replay["decode"]()
        e2.record()
        evs.append((e0, e1, e2))
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_wall = time.perf_counter() - t_wall0
    step_ms = [a.elapsed_time(c) for a, _, c in evs]
    dec_ms = [b.elapsed_time(c) for _, b, c in evs]
    pre_ms = [a.elapsed_time(b) for a, b, _ in evs]

    # the dominant kernel alone (partition kernel), for the roofline: `steps`
    # launches back to back between one pair of events, so that the average
    # launch duration excludes the graph-launch gap before each one (each
    # launch streams inputs larger than L2; with --flush write a flush runs
    # between launches and is timed per launch instead)
    part_ms = []
    if args.flush != "none":
        for i in range(args.steps):
            maybe_flush(i)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            replay["partitions"]()
            b.record()
            part_ms.append((a, b))
        torch.cuda.synchronize()
        part_ms = [a.elapsed_time(b) for a, b in part_ms]
    else:
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(args.steps):
            replay["partitions"]()
        b.record()
        torch.cuda.synchronize()
        part_ms = [a.elapsed_time(b) / args.steps] * args.steps

    # the same kernel launched alone after a 512 MiB read of another buffer
    # (L2 then holds none of the call's lines, all clean), timed per launch:
    # what a launch costs with nothing of it left in L2 and no overlap with
    # a launch before it
    cold = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    cold_sink = torch.zeros(1, dtype=torch.int64, device=dev)
    cold_ms = []
    for i in range(args.steps):
        cold_sink.add_(cold.view(torch.int64).sum())
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        replay["partitions"]()
        b.record()
        cold_ms.append((a, b))
    torch.cuda.synchronize()
    cold_ms = [a.elapsed_time(b) for a, b in cold_ms]
    del cold

    # the step again as ONE graph (copy, append and decode captured
    # together, event nodes between them): the decode call's interval then
    # holds no graph launch, as in an engine that captures its whole step
    one_graph = None
    timer = step_graph(stream, [pre, decode]) if not args.no_graphs else None
    if timer is not None:
        for i in range(args.warmup):
            maybe_flush(i)
            timer()
        one_graph = []
        for i in range(args.steps):
            maybe_flush(i)
            one_graph.append(timer())
    clk = clocks.stop() if clocks else None

    # two graphs per step (the copy-and-append graph, then the decode graph)
    sep_dec_s, sep_step_s = slowest([sum(dec_ms) / 1e3, sum(step_ms) / 1e3], dev)
    if one_graph is not None:
        pre_ms = [a for a, _ in one_graph]
        dec_ms = [b for _, b in one_graph]
        step_ms = [a + b for a, b in one_graph]
    dec_s = sum(dec_ms) / 1e3
    step_s = sum(step_ms) / 1e3
    dbytes = w.decode_bytes()
    dec_s, step_s = slowest([dec_s, step_s], dev)
    # bytes the decode call must read: with shared prefixes every distinct
    # block once (the prefix is read once per group), else every sequence's
    # K/V; `value` counts these, never a shared block once per member
    rbytes = dbytes - w.kv_bytes() + w.unique_kv_bytes() if shared else dbytes
    value = whole_job_rate(rbytes * args.steps, dec_s, world) / 1e9

    # end to end through the C ABI from pinned host buffers: the step's
    # inputs are packed into one pinned staging buffer and cross with one
    # host-to-device copy; the output comes back with one device-to-host copy
    e2e = None
    if not args.no_e2e:
        host_in = [("q", np.ascontiguousarray(w.q), iodt), ("k", np.ascontiguousarray(sk), iodt),
                   ("v", np.ascontiguousarray(sv), iodt), ("slots", w.step_slots, torch.int64),
                   ("bt", w.block_tables, torch.int32), ("cl", w.context_lens, torch.int32)]
        if pairs is not None:
            host_in.append(("pairs", w.copy_pairs, torch.int64))
        if shared:
            host_in += [("gb", grp_begin, torch.int32), ("gp", grp_blocks, torch.int32)]
        offs, total = {}, 0
        for name, arr, _ in host_in:
            offs[name] = total
            total += -(-arr.nbytes // 256) * 256
        h_stage = torch.empty(total, dtype=torch.uint8).pin_memory()
        d_stage = torch.empty(total, dtype=torch.uint8, device=dev)
        views = {}
        for name, arr, dt in host_in:
            o, nb = offs[name], arr.nbytes
            h_stage[o:o + nb].copy_(torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8)
                                                     .reshape(-1)))
            views[name] = d_stage[o:o + nb].view(dt).view(arr.shape)
        h_out = torch.empty(out.shape, dtype=iodt).pin_memory()
        h2d, d2h = total, h_out.numel() * h_out.element_size()

        def step_e2e():
            if pairs is not None:
                B.pkv_copy_blocks(desc, views["pairs"])
            B.pkv_kv_append(desc, views["k"], views["v"], views["slots"])
            if shared:
                B.pkv_paged_attention_decode_shared_prefix(
                    desc, views["q"], views["bt"], views["cl"], w.max_context_len, views["gb"],
                    views["gp"], max_group, max_prefix, w.scale, partition_size=shared_ps,
                    workspace=workspace, out=out)
            else:
                B.pkv_paged_attention_decode(desc, views["q"], views["bt"], views["cl"],
                                             w.max_context_len, w.scale, partition_size=ps,
                                             workspace=workspace, out=out)

        def e2e_once():
            d_stage.copy_(h_stage, non_blocking=True)
            step_e2e()
            h_out.copy_(out, non_blocking=True)

        def time_e2e(run):
            ms = []
            for i in range(args.steps + args.warmup):
                maybe_flush(i)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record()
                run()
                b.record()
                b.synchronize()
                if i >= args.warmup:
                    ms.append(a.elapsed_time(b))
            sec = slowest([sum(ms) / 1e3], dev)[0]
            return {"value": whole_job_rate(rbytes * args.steps, sec, world) / 1e9,
                    "ms_per_step": sec * 1e3 / args.steps}

        # every step runs the C-ABI host code (argument checks, partition
        # choice, launches) between the events, as a caller's step does
        direct = time_e2e(e2e_once)
        e2e = {"value": direct["value"], "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": direct["ms_per_step"],
               "timing": "per step, between CUDA events: the pinned host-to-device copy of "
                         "the packed inputs, the C-ABI calls made from Python (host checks "
                         "and kernel launches included), the device-to-host copy of out"}
        if not args.no_graphs:
            # the same copies and C-ABI launches captured once into a CUDA
            # graph: a replay runs the kernels and copies only (the calls'
            # host code ran at capture)
            e2e_once()
            torch.cuda.synchronize()
            ge = torch.cuda.CUDAGraph()
            with torch.cuda.graph(ge, stream=stream):
                e2e_once()
            torch.cuda.synchronize()
            gr = time_e2e(ge.replay)
            e2e["graph_replay"] = {
                "value": gr["value"], "unit": "GB/s", "ms_per_step": gr["ms_per_step"],
                "timing": "graph replay of the captured C-ABI launches (copies and kernels "
                          "only; no host code of the calls in the timed region)"}

    peak, peak_kind = hbm_peak()
    part_mean = sum(part_ms) / len(part_ms) / 1e3
    achieved = rbytes / part_mean / 1e9
    tr = NCU_TRAFFIC.get(w.name + (":shared-prefix" if shared else ""))
    traffic = tr["bytes_per_launch"] if tr and tr.get("src_sha") == decode_src_sha() else None
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic,
                "traffic_source": tr.get("profile") if tr and traffic is not None else None,
                "kernel": ("shared-prefix decode call, single pass: decode_group_kernel"
                           if single else
                           "shared-prefix decode call: decode_mma_kernel over the prefixes, "
                           + decode_kernel_name(w) + " over the rest, lse_reduce_kernel"
                           if shared else
                           decode_kernel_name(w) + " (pkv_paged_attention_partitions)"),
                "algorithmic_bytes": rbytes,
                "frac_alone_after_l2_read": rbytes / (statistics.mean(cold_ms) / 1e3) / 1e9 / peak,
                "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s"}

    # the workload's config, the same in the reference arm's line; how this
    # arm measured it goes under "measurement"
    cfg = workload_config(w)
    if args.flush != "none":
        cfg["l2"] = ("512 MiB %s between steps (L2 flush)"
                     % ("written" if args.flush == "write" else "read"))
    measurement = {}
    measurement["timing"] = (("value: the decode call between event nodes inside one CUDA graph of "
                      "the whole step (copy, append, decode); separate_graphs: the same "
                      "with the step as two graphs, events between their replays; "
                      if one_graph is not None else
                      "value: CUDA events around CUDA-graph replays of the decode call; ")
                     + "roofline: the partition kernel launched `steps` times back to back "
                     "between one pair of events; e2e: see e2e.timing") \
        if not args.no_graphs else "CUDA events around direct calls"
    measurement["partition_size"] = ps
    measurement["shared_prefix"] = ({"groups": int(len(grp_blocks)), "max_group": max_group,
                                     "prefix_blocks": max_prefix,
                                     "route": "single pass" if single else "split"}
                                    if shared else None)
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_s * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": cfg, "measurement": measurement,
            "hbm_frac": value / peak,
            "decode_ms": dec_s * 1e3 / args.steps,
            "decode_tokens_per_s": w.num_seqs * world * args.steps / dec_s,
            "model_tokens_per_s_attention_only":
                w.num_seqs * world * args.steps / dec_s / MODEL_LAYERS.get(w.name, 1),
            "step_ms": {"copy_and_append": statistics.mean(pre_ms),
                        "decode": statistics.mean(dec_ms), "step": statistics.mean(step_ms)},
            "decode_ms_spread": percentiles(dec_ms),
            "separate_graphs": {"value": whole_job_rate(rbytes * args.steps, sep_dec_s,
                                                        world) / 1e9,
                                "decode_ms": sep_dec_s * 1e3 / args.steps,
                                "step_ms": sep_step_s * 1e3 / args.steps},
            "decode_bytes": dbytes, "unique_kv_bytes": w.unique_kv_bytes(),
            "roofline": roofline, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk, "wall_s": t_wall}
    if w.unique_kv_bytes() != w.kv_bytes():
        # shared prompt blocks: every sequence's K/V counted in full (a shared
        # block once per member), the decode's logical work
        line["logical_bytes_gbs"] = dbytes * args.steps * world / dec_s / 1e9
    del replay, stages
    if world > 1:
        dist.barrier()
    if rank == 0 and not args.no_cpu_baseline:
        cand = None if sample_cap_bytes is None else sample_sequences(w, sample_cap_bytes)
        hs = HostState(w, seqs=cand, threads=threads)
        seqs, reps = pick_sample(w, cpu_budget_s, hs, cand)
        t = oracle_decode_sample(w, hs, seqs, reps)
        line["cpu_baseline"] = {
            "value": sample_bytes(w, seqs) * reps / t / 1e9, "unit": "GB/s",
            "cores": os.cpu_count() or 1, "kind": "oracle",
            "sample": "oracle decode of %d of %d sequences x %d repetitions (%d context tokens "
                      "each), fp64, all host threads" % (len(seqs), w.num_seqs, reps,
                                                        int(w.context_lens[seqs].sum()))}
    return line if rank == 0 else None


# the other decode workloads of the default run, each timed like the headline
EXTRA_CONFIGS = ("llama2_70b_bf16_gqa", "cow_parallel_sampling_f16", "llama2_7b_fp8_long")
# host K/V a config's bounded oracle sample is drawn from (the E4M3 layer
# holds 2.5 GB; drawing all of it again for the CPU baseline would take minutes)
EXTRA_SAMPLE_CAP = 400 << 20


def config_summary(line):
    """The per-config entry of the default run's `configs` key."""
    keep = ("value", "unit", "hbm_frac", "decode_ms", "ms_per_step", "decode_tokens_per_s",
            "model_tokens_per_s_attention_only", "decode_ms_spread", "decode_bytes",
            "unique_kv_bytes", "logical_bytes_gbs", "roofline", "e2e", "gpu_launches", "clocks",
            "cpu_baseline", "config", "measurement")
    return {k: line[k] for k in keep if k in line}


# ------------------------------------------------------------------ prefill arm

PREFILL_METRIC = "paged prefill attention TFLOP/s (causal, new tokens over the paged cache)"


def prefill_oracle_rows(w, hs, rows):
    """Time the oracle's prefill of query `rows` (each the decode of its
    position's causal context); returns (seconds, flops of those rows)."""
    import oracle
    cu = w.cu_seqlens_q.astype(np.int64)
    seq = np.searchsorted(cu, rows, side="right") - 1
    n = cu[seq + 1] - cu[seq]
    pos = w.context_lens[seq].astype(np.int64) - n + (rows - cu[seq])
    t0 = time.perf_counter()
    oracle.paged_attention_decode(hs.k_cache, hs.v_cache, w.cache_dtype, w.q[rows], w.io_dtype,
                                  w.block_tables[seq], (pos + 1).astype(np.int32), w.scale)
    t = time.perf_counter() - t0
    return t, int(4 * (pos + 1).sum() * w.head_dim * w.num_heads)


def prefill_cpu_sample(w, hs, budget_s):
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(w.total_q, min(w.total_q, 16), replace=False))
    t, f = prefill_oracle_rows(w, hs, rows)
    n = int(min(w.total_q, max(16, len(rows) * budget_s / max(t, 1e-3))))
    rows = np.sort(rng.choice(w.total_q, n, replace=False))
    return rows


def run_reference_prefill(args, w, prefill):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    hs = HostState(w, prefill)
    cores = os.cpu_count() or 1
    rows = prefill_cpu_sample(w, hs, 20.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        prefill_oracle_rows(w, hs, rows)
    tot_t, tot_f = 0.0, 0
    for _ in range(args.steps):
        t, f = prefill_oracle_rows(w, hs, rows)
        tot_t += t
        tot_f += f
    v = tot_f / tot_t / 1e12
    return {"metric": PREFILL_METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot_t * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference", "config": prefill_config(w),
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": "%d of %d query rows per step" % (len(rows), w.total_q)},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def prefill_traffic(w):
    """DRAM bytes per launch from the ncu capture, while the prefill sources
    are unchanged since (else None)."""
    tr = NCU_PREFILL_TRAFFIC.get(w.name)
    return tr["bytes_per_launch"] if tr and tr["src_sha"] == src_sha(PREFILL_SOURCES) else None


def hash_traffic(w):
    """DRAM bytes per launch from the ncu capture, while the hash kernel's
    sources are unchanged since (else None)."""
    tr = NCU_HASH_TRAFFIC.get(w.name)
    return tr["bytes_per_launch"] if tr and tr["src_sha"] == src_sha(HASH_SOURCES) else None


def prefill_config(w):
    cfg = workload_config(w)
    cfg.update({"new_tokens": w.total_q, "max_q_len": w.max_q_len,
                "cached_tokens": int(w.context_lens.sum()) - w.total_q,
                "l2": "K/V of the batch (%.0f MB) are read once per CTA (two 128-row "
                      "query tiles); compute-bound, no flush" % (w.kv_bytes() / 1e6)})
    return cfg


def run_gpu_prefill(args, w, prefill):
    import torch
    import torch.distributed as dist
    from paged_kv_cache_130_gb300 import binding as B
    from paged_kv_cache_130_gb300 import build as pkv_build

    world, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=dev)
    pkv_build.build()
    B.load()
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    dt = {0: torch.float16, 1: torch.bfloat16}[w.io_dtype]
    k_cache = torch.zeros(shape, dtype=dt, device=dev)
    v_cache = torch.zeros(shape, dtype=dt, device=dev)
    desc = B.cache_desc(k_cache, v_cache)

    def dev16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(dt).to(dev)

    for slots, k, v in prefill:
        B.pkv_kv_append(desc, dev16(k), dev16(v), torch.from_numpy(slots).to(dev))
    sk, sv = w.step_values()
    step_k, step_v = dev16(sk), dev16(sv)
    step_slots = torch.from_numpy(w.step_slots).to(dev)
    q = dev16(w.q)
    cu = torch.from_numpy(w.cu_seqlens_q).to(dev)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    out = torch.empty_like(q)
    flops = w.prefill_flops()

    def pre():
        B.pkv_kv_append(desc, step_k, step_v, step_slots)

    def attn():
        B.pkv_paged_attention_prefill(desc, q, cu, w.max_q_len, bt, cl, w.max_context_len,
                                      w.scale, out=out)

    for _ in range(args.warmup):
        pre()
        attn()
    torch.cuda.synchronize()
    replay = {"pre": pre, "attn": attn}
    if not args.no_graphs:
        for name, fn in list(replay.items()):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            replay[name] = g.replay
        torch.cuda.synchronize()
    clocks = ClockSampler(local) if not args.no_clocks else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    evs = []
    for _ in range(args.steps):
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record()
        replay["pre"]()
        e1.record()
        replay["attn"]()
        e2.record()
        evs.append((e0, e1, e2))
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    attn_s = sum(b.elapsed_time(c) for _, b, c in evs) / 1e3
    step_s = sum(a.elapsed_time(c) for a, _, c in evs) / 1e3
    attn_s, step_s = slowest([attn_s, step_s], dev)
    value = whole_job_rate(flops * args.steps, attn_s, world) / 1e12

    e2e = None
    if not args.no_e2e:
        h = {"q": w.q, "k": sk, "v": sv}
        hq, hk, hv = (torch.from_numpy(np.ascontiguousarray(h[x]).view(np.int16)).view(dt)
                      .pin_memory() for x in ("q", "k", "v"))
        hslots = torch.from_numpy(w.step_slots).pin_memory()
        hcu = torch.from_numpy(w.cu_seqlens_q).pin_memory()
        hbt = torch.from_numpy(w.block_tables).pin_memory()
        hcl = torch.from_numpy(w.context_lens).pin_memory()
        hout = torch.empty(out.shape, dtype=dt).pin_memory()
        ins = (hq, hk, hv, hslots, hcu, hbt, hcl)
        h2d = sum(t.numel() * t.element_size() for t in ins)
        d2h = hout.numel() * hout.element_size()
        ms = []
        for i in range(args.steps + args.warmup):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            for dst, src in zip((q, step_k, step_v, step_slots, cu, bt, cl), ins):
                dst.copy_(src, non_blocking=True)
            pre()
            attn()
            hout.copy_(out, non_blocking=True)
            b.record()
            b.synchronize()
            if i >= args.warmup:
                ms.append(a.elapsed_time(b))
        e2e_s = slowest([sum(ms) / 1e3], dev)[0]
        e2e = {"value": whole_job_rate(flops * args.steps, e2e_s, world) / 1e12,
               "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_s * 1e3 / args.steps}

    # the kernel alone for the roofline: `steps` launches back to back
    ra = torch.cuda.Event(enable_timing=True)
    rb = torch.cuda.Event(enable_timing=True)
    ra.record()
    for _ in range(args.steps):
        replay["attn"]()
    rb.record()
    torch.cuda.synchronize()
    peak, kind = tensor_peak()
    achieved = flops / (ra.elapsed_time(rb) / 1e3 / args.steps) / 1e12
    line = {"metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_s * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": {0: "f16", 1: "bf16"}[w.io_dtype], "data": "synthetic",
            "config": prefill_config(w),
            "prefill_flops": flops,
            "step_ms": {"append": sum(a.elapsed_time(b) for a, b, _ in evs) / args.steps,
                        "prefill": attn_s * 1e3 / args.steps},
            "prefill_ms_spread": percentiles([b.elapsed_time(c) for _, b, c in evs]),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "traffic": prefill_traffic(w),
                         "kernel": "prefill_ws_kernel (pkv_paged_attention_prefill)",
                         "peak_source": kind + " (MEASURED_PEAKS.json bf16_tflops, burst)"
                         if kind == "measured" else "fallback 1.9 PFLOP/s"},
            "e2e": e2e, "gpu_launches": 2 * args.steps, "clocks": clk}
    if rank == 0 and not args.no_cpu_baseline:
        hs = HostState(w, prefill)
        rows = prefill_cpu_sample(w, hs, 15.0)
        t, f = prefill_oracle_rows(w, hs, rows)
        line["cpu_baseline"] = {"value": f / t / 1e12, "unit": "TFLOP/s",
                                "cores": os.cpu_count() or 1, "kind": "oracle",
                                "sample": "%d of %d query rows" % (len(rows), w.total_q)}
    return line if rank == 0 else None


# ------------------------------------------------------------------ swap arm

SWAP_METRIC = "block swap GB/s (device cache <-> pinned host memory, out + in)"


def swap_oracle_sample(w, layers=2):
    """Oracle swap of `layers` layers of the workload on host arrays; returns
    (seconds, bytes moved)."""
    import oracle
    shape = (w.num_kv_heads, w.block_size, w.head_dim)
    dk = [np.full((w.num_blocks,) + shape, l + 1, np.uint16) for l in range(layers)]
    dv = [np.full((w.num_blocks,) + shape, l + 2, np.uint16) for l in range(layers)]
    # written before the clock starts, so that first-touch page faults stay out
    hk = [np.full((w.host_blocks,) + shape, 0, np.uint16) for _ in range(layers)]
    hv = [np.full((w.host_blocks,) + shape, 0, np.uint16) for _ in range(layers)]
    t0 = time.perf_counter()
    oracle.swap_blocks(dk, dv, hk, hv, w.out_pairs)
    oracle.swap_blocks(hk, hv, dk, dv, w.in_pairs)
    t = time.perf_counter() - t0
    return t, w.swap_bytes() * layers // w.num_layers


def swap_config(w):
    return {"workload": w.name, "num_layers": w.num_layers, "num_blocks": w.num_blocks,
            "host_blocks": w.host_blocks, "num_kv_heads": w.num_kv_heads,
            "block_size": w.block_size, "head_dim": w.head_dim, "cache_dtype": "f16",
            "swapped_sequences": int(len(w.swapped_seqs)), "pairs_each_way": int(len(w.out_pairs)),
            "block_bytes": w.block_bytes,
            "l2": "%.1f GB moved per step exceeds the 129 MB L2" % (w.swap_bytes() / 1e9),
            "parallelism": "replicas"}


def run_reference_swap(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    for _ in range(args.warmup):
        swap_oracle_sample(w)
    tt, bb = 0.0, 0
    for _ in range(args.steps):
        t, b = swap_oracle_sample(w)
        tt += t
        bb += b
    v = bb / tt / 1e9
    return {"metric": SWAP_METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
            "data": "synthetic", "impl": "reference", "config": swap_config(w),
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "2 of %d layers per step" % w.num_layers},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_gpu_swap(args, w):
    import torch
    import torch.distributed as dist
    from paged_kv_cache_130_gb300 import binding as B
    from paged_kv_cache_130_gb300 import build as pkv_build

    world, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=dev)
    pkv_build.build()
    B.load()
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    shape = (w.num_kv_heads, w.block_size, w.head_dim)
    dk = [torch.full((w.num_blocks,) + shape, float(l), dtype=torch.float16, device=dev)
          for l in range(w.num_layers)]
    dv = [torch.full((w.num_blocks,) + shape, -float(l), dtype=torch.float16, device=dev)
          for l in range(w.num_layers)]
    hk = [torch.empty((w.host_blocks,) + shape, dtype=torch.float16).pin_memory()
          for _ in range(w.num_layers)]
    hv = [torch.empty((w.host_blocks,) + shape, dtype=torch.float16).pin_memory()
          for _ in range(w.num_layers)]
    ddesc = [B.cache_desc(a, b) for a, b in zip(dk, dv)]
    hdesc = [B.cache_desc(a, b) for a, b in zip(hk, hv)]
    p_out = torch.from_numpy(w.out_pairs).to(dev)
    p_in = torch.from_numpy(w.in_pairs).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def out():
        B.pkv_swap_blocks(ddesc, hdesc, p_out, dev_err=err)

    def back():
        B.pkv_swap_blocks(hdesc, ddesc, p_in, dev_err=err)

    for _ in range(args.warmup):
        out()
        back()
    torch.cuda.synchronize()
    clocks = ClockSampler(local) if not args.no_clocks else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    evs = []
    for _ in range(args.steps):
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record()
        out()
        e1.record()
        back()
        e2.record()
        evs.append((e0, e1, e2))
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    out_s = sum(a.elapsed_time(b) for a, b, _ in evs) / 1e3
    in_s = sum(b.elapsed_time(c) for _, b, c in evs) / 1e3
    out_s, in_s = slowest([out_s, in_s], dev)
    moved = w.swap_bytes()
    value = whole_job_rate(moved * args.steps, out_s + in_s, world) / 1e9

    # The link's measured ceiling for this run, each way, on one 2 GiB pinned
    # buffer: the copy engines (cudaMemcpyAsync) and an SM-driven streaming
    # copy (pkv_testing_stream_copy: plain loads and stores over NVLink-C2C,
    # the path the swap kernel takes); the better of the two per direction
    nbytes = 2 << 30
    dbuf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    hbuf = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    link = {}
    for how in ("copy_engine", "sm_stream"):
        for direction in ("d2h", "h2d"):
            best = 0.0
            for _ in range(3):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                dst, src = (hbuf, dbuf) if direction == "d2h" else (dbuf, hbuf)
                a.record()
                if how == "copy_engine":
                    dst.copy_(src, non_blocking=True)
                else:
                    B.pkv_testing_stream_copy(dst, src)
                b.record()
                b.synchronize()
                best = max(best, nbytes / (a.elapsed_time(b) / 1e3) / 1e9)
            link[how + "_" + direction] = best
    rates = [max(link["copy_engine_d2h"], link["sm_stream_d2h"]),
             max(link["copy_engine_h2d"], link["sm_stream_h2d"])]
    peak = 2.0 / (1.0 / rates[0] + 1.0 / rates[1])      # out and in take equal bytes
    del dbuf, hbuf

    e2e = None
    if not args.no_e2e:
        hp_out = torch.from_numpy(w.out_pairs).pin_memory()
        hp_in = torch.from_numpy(w.in_pairs).pin_memory()
        herr = torch.zeros(1, dtype=torch.int32).pin_memory()
        ms = []
        for i in range(args.steps + args.warmup):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            p_out.copy_(hp_out, non_blocking=True)
            p_in.copy_(hp_in, non_blocking=True)
            out()
            back()
            herr.copy_(err, non_blocking=True)
            b.record()
            b.synchronize()
            if i >= args.warmup:
                ms.append(a.elapsed_time(b))
        e2e_s = slowest([sum(ms) / 1e3], dev)[0]
        e2e = {"value": whole_job_rate(moved * args.steps, e2e_s, world) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": int(moved // 2 + 16 * len(w.out_pairs)),
               "d2h_bytes_per_step": int(moved // 2 + 4),
               "ms_per_step": e2e_s * 1e3 / args.steps}
    line = {"metric": SWAP_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": (out_s + in_s) * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": swap_config(w), "swap_bytes_per_step": moved,
            "step_ms": {"out": out_s * 1e3 / args.steps, "in": in_s * 1e3 / args.steps},
            "roofline": {"bound": "c2c", "achieved": value, "peak": peak, "unit": "GB/s",
                         "frac": value / peak, "traffic": None,
                         "kernel": "swap_blocks_kernel (pkv_swap_blocks, both directions)",
                         "peak_source": "measured in this run on 2 GiB pinned, the better of "
                                        "the copy engines and an SM streaming copy each way: "
                                        "D2H %.0f GB/s, H2D %.0f GB/s" % tuple(rates),
                         "link_gbs": link},
            "e2e": e2e, "gpu_launches": 2 * args.steps, "clocks": clk,
            "dev_err": int(err.item())}
    if rank == 0 and not args.no_cpu_baseline:
        t, b = swap_oracle_sample(w)
        line["cpu_baseline"] = {"value": b / t / 1e9, "unit": "GB/s", "cores": 1,
                                "kind": "oracle", "sample": "2 of %d layers" % w.num_layers}
    return line if rank == 0 else None


# ------------------------------------------------------------------ hash arm

HASH_METRIC = "prefix-cache block hashing GB/s (token bytes through chained SHA-256)"
# integer operations of one SHA-256 compression: 64 rounds of ~22 and 48
# message-schedule steps of ~12 (a rotate counts as one funnel shift)
SHA256_OPS = 64 * 22 + 48 * 12


# The SHA-256 round's longest dependency (e_i -> e_{i+1}): the rotations of
# Sigma1, their three-way XOR, one three-input add of the terms that were
# ready earlier -- three dependent integer operations of about four cycles.
INT_OP_LATENCY = 4
CYCLES_PER_ROUND = 3 * INT_OP_LATENCY


def hash_chunks(w):
    return (4 * (8 + w.block_size) + 9 + 63) // 64


def hash_chain_bound(w, sm_mhz=2070.0):
    """Token GB/s if the longest chain of block hashes ran at the SHA-256
    round's dependency latency (the chain is sequential by definition, so
    the launch cannot end before it): hashed bytes / that chain's time.
    Returns (GB/s, blocks of the longest chain)."""
    lens = np.diff(w.cu_seqlens.astype(np.int64))
    chain = int((lens // w.block_size).max(initial=0))
    cycles = chain * hash_chunks(w) * 64 * CYCLES_PER_ROUND
    t = cycles / (sm_mhz * 1e6)
    return (w.hashed_token_bytes() / t / 1e9 if t > 0 else 0.0), chain


def hash_alu_peak(w, sm_mhz=2070.0):
    """Token GB/s if every INT32 lane of the GPU ran compressions: 152 SMs x
    128 lanes x clock, / the operations of one block, x its token bytes."""
    nch = (4 * (8 + w.block_size) + 9 + 63) // 64
    ops = 152 * 128 * sm_mhz * 1e6
    return ops / (nch * SHA256_OPS) * 4 * w.block_size / 1e9


def hash_oracle_sample(w, seqs):
    import oracle
    cu = w.cu_seqlens.astype(np.int64)
    toks = w.token_ids[cu[seqs[0]]:cu[seqs[-1] + 1]]
    sub = np.concatenate([[0], np.cumsum(np.diff(cu)[seqs])])
    t0 = time.perf_counter()
    oracle.block_hashes(toks, sub, w.block_size)
    t = time.perf_counter() - t0
    full = int((np.diff(sub) // w.block_size).sum())
    return t, 4 * w.block_size * full


def hash_config(w):
    return {"workload": w.name, "num_seqs": w.num_seqs, "block_size": w.block_size,
            "tokens": int(len(w.token_ids)), "full_blocks": w.full_blocks(),
            "hash": "SHA-256(parent hash || token ids as little-endian int32)",
            "l2": "token ids (%.0f MB) are read once" % (len(w.token_ids) * 4 / 1e6),
            "parallelism": "replicas"}


def run_reference_hash(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    seqs = np.arange(min(w.num_seqs, 256))
    for _ in range(args.warmup):
        hash_oracle_sample(w, seqs)
    tt, bb = 0.0, 0
    for _ in range(args.steps):
        t, b = hash_oracle_sample(w, seqs)
        tt += t
        bb += b
    v = bb / tt / 1e9
    return {"metric": HASH_METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
            "data": "synthetic", "impl": "reference", "config": hash_config(w),
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "%d of %d sequences per step" % (len(seqs), w.num_seqs)},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_gpu_hash(args, w):
    import torch
    import torch.distributed as dist
    from paged_kv_cache_130_gb300 import binding as B
    from paged_kv_cache_130_gb300 import build as pkv_build

    world, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=dev)
    pkv_build.build()
    B.load()
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    toks = torch.from_numpy(w.token_ids).to(dev)
    cu = torch.from_numpy(w.cu_seqlens).to(dev)
    full = np.diff(w.cu_seqlens.astype(np.int64)) // w.block_size
    offs = torch.from_numpy(np.cumsum(full) - full).to(dev)
    nblk = w.full_blocks()
    hashes = torch.empty((nblk, 32), dtype=torch.uint8, device=dev)

    def run():
        B.pkv_block_hashes(toks, cu, w.block_size, block_offsets=offs, hashes=hashes)

    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    clocks = ClockSampler(local) if not args.no_clocks else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    evs = []
    for _ in range(args.steps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        run()
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    t = slowest([sum(a.elapsed_time(b) for a, b in evs) / 1e3], dev)[0]
    nbytes = w.hashed_token_bytes()
    value = whole_job_rate(nbytes * args.steps, t, world) / 1e9
    e2e = None
    if not args.no_e2e:
        ht = torch.from_numpy(w.token_ids).pin_memory()
        hcu = torch.from_numpy(w.cu_seqlens).pin_memory()
        hoff = offs.cpu().pin_memory()
        hh = torch.empty(hashes.shape, dtype=torch.uint8).pin_memory()
        ms = []
        for i in range(args.steps + args.warmup):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            toks.copy_(ht, non_blocking=True)
            cu.copy_(hcu, non_blocking=True)
            offs.copy_(hoff, non_blocking=True)
            run()
            hh.copy_(hashes, non_blocking=True)
            b.record()
            b.synchronize()
            if i >= args.warmup:
                ms.append(a.elapsed_time(b))
        e2e_s = slowest([sum(ms) / 1e3], dev)[0]
        e2e = {"value": whole_job_rate(nbytes * args.steps, e2e_s, world) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": int(4 * (len(w.token_ids) + len(w.cu_seqlens))
                                         + 8 * w.num_seqs),
               "d2h_bytes_per_step": int(32 * nblk), "ms_per_step": e2e_s * 1e3 / args.steps}
    sm_mhz = clk["sm_mhz"] if clk else 2070.0
    peak, chain = hash_chain_bound(w, sm_mhz)
    line = {"metric": HASH_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
            "data": "synthetic", "config": hash_config(w),
            "roofline": {"bound": "latency", "achieved": value, "peak": peak, "unit": "GB/s",
                         "frac": value / peak, "traffic": hash_traffic(w),
                         "kernel": "block_hash_kernel (pkv_block_hashes)",
                         "peak_source": "derived chain-latency bound: the longest chain, %d "
                                        "blocks x %d compressions x 64 rounds x %d cycles a "
                                        "round (%d dependent integer operations of ~%d "
                                        "cycles), at %.0f MHz" % (
                                            chain, hash_chunks(w), CYCLES_PER_ROUND,
                                            CYCLES_PER_ROUND // INT_OP_LATENCY,
                                            INT_OP_LATENCY, sm_mhz),
                         "alu_width_peak": hash_alu_peak(w, sm_mhz)},
            "e2e": e2e, "gpu_launches": args.steps, "clocks": clk}
    if rank == 0 and not args.no_cpu_baseline:
        tt, bb = hash_oracle_sample(w, np.arange(min(w.num_seqs, 256)))
        line["cpu_baseline"] = {"value": bb / tt / 1e9, "unit": "GB/s", "cores": 1,
                                "kind": "oracle", "sample": "256 of %d sequences" % w.num_seqs}
    return line if rank == 0 else None


def main(argv=None):
    args = parse_args(argv)
    from paged_kv_cache_130_gb300 import workloads as W
    world, rank, local = dist_env()
    if args.impl == "reference" and rank != 0:
        return 0
    w = W.make(args.workload) if args.num_seqs is None else \
        W.make(args.workload, num_seqs=args.num_seqs)
    if isinstance(w, W.HashWorkload):
        line = (run_reference_hash if args.impl == "reference" else run_gpu_hash)(args, w)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    if isinstance(w, W.SwapWorkload):
        line = (run_reference_swap if args.impl == "reference" else run_gpu_swap)(args, w)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    if w.cu_seqlens_q is not None:
        prefill = list(w.prefill())
        run = run_reference_prefill if args.impl == "reference" else run_gpu_prefill
        line = run(args, w, prefill)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    if args.impl == "reference":
        line = run_reference(args, w)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0

    import torch
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    line = run_gpu(args, w)
    extra = ()
    if args.configs == "auto":
        extra = EXTRA_CONFIGS if args.workload == DEFAULT_WORKLOAD and args.num_seqs is None \
            else ()
    elif args.configs != "none":
        extra = tuple(n for n in args.configs.split(",") if n and n != args.workload)
    if extra:
        configs = {w.name: config_summary(line) if line is not None else None}
        for name in extra:
            torch.cuda.empty_cache()
            w2 = W.make(name)
            line2 = run_gpu(args, w2, cpu_budget_s=4.0, sample_cap_bytes=EXTRA_SAMPLE_CAP)
            if line2 is not None:
                configs[name] = config_summary(line2)
            del w2
        if line is not None:
            line["configs"] = configs
    if world > 1 and dist.is_initialized():
        dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
