"""Host-side pieces of bench.py that need no GPU: the bounded oracle sample
of a workload, the per-config summary, and the options."""
import numpy as np

import bench
from paged_kv_cache_130_gb300 import workloads as W


def test_sample_sequences_fit_the_cap():
    w = W.llama2_70b_bf16_gqa(num_seqs=8)
    per = w.context_lens.astype(np.int64) * w.num_kv_heads * w.head_dim * 2 * 2
    for cap in (1, int(per[0]), int(per[:3].sum()), 1 << 40):
        seqs = bench.sample_sequences(w, cap)
        assert len(seqs) >= 1 and list(seqs) == list(range(len(seqs)))
        if len(seqs) > 1:
            assert per[:len(seqs)].sum() <= cap
        if len(seqs) < w.num_seqs:
            assert per[:len(seqs) + 1].sum() > cap


def test_host_state_of_a_sample_matches_the_whole_on_its_blocks():
    """The oracle's caches built from the sampled sequences' segments alone
    hold the same bytes in those sequences' blocks as the whole build."""
    for w in (W.tiny_f16(), W.cow_parallel_sampling_f16(num_prompts=3, samples=3,
                                                         prompt_len=40, tail_hi=20,
                                                         num_heads=4, head_dim=64)):
        whole = bench.HostState(w)
        seqs = [1, 2]
        part = bench.HostState(w, seqs=seqs, threads=2)
        for s in seqs:
            nblk = -(-int(w.context_lens[s]) // w.block_size)
            blocks = w.block_tables[s, :nblk]
            assert np.array_equal(part.k_cache[blocks], whole.k_cache[blocks])
            assert np.array_equal(part.v_cache[blocks], whole.v_cache[blocks])


def test_threaded_prefill_draws_the_same_values():
    w = W.opt13b_f16(num_seqs=3)
    one = list(w.prefill())
    many = list(w.prefill(threads=3))
    assert len(one) == len(many)
    for (s1, k1, v1), (s2, k2, v2) in zip(one, many):
        assert np.array_equal(s1, s2) and np.array_equal(k1, k2) and np.array_equal(v1, v2)


def test_fp8_scale_calibration_does_not_depend_on_threads():
    a = W.llama2_7b_fp8_long(num_seqs=2, lo=300, hi=900, calibrate=False)
    a.calibrate_fp8_scales(threads=1)
    b = W.llama2_7b_fp8_long(num_seqs=2, lo=300, hi=900, calibrate=False)
    b.calibrate_fp8_scales(threads=4)
    assert (a.k_scale, a.v_scale) == (b.k_scale, b.v_scale)
    # the scale is amax / 448 of every value written, K and V apart
    amax = 0.0
    for _, k, _ in a.prefill():
        amax = max(amax, float(np.abs(W.bits_to_float32(k, a.io_dtype)).max()))
    k, _ = a.step_values()
    amax = max(amax, float(np.abs(W.bits_to_float32(k, a.io_dtype)).max()))
    assert a.k_scale == float(np.float32(amax) / np.float32(448.0))


def test_config_summary_and_options():
    line = {"value": 1.0, "unit": "GB/s", "roofline": {"frac": 0.5}, "clocks": None,
            "config": {"workload": "x"}, "metric": "m", "steps": 3}
    got = bench.config_summary(line)
    assert got == {"value": 1.0, "unit": "GB/s", "roofline": {"frac": 0.5}, "clocks": None,
                   "config": {"workload": "x"}}
    assert bench.parse_args([]).configs == "auto"
    assert bench.parse_args(["--configs", "none"]).configs == "none"
    assert set(bench.EXTRA_CONFIGS) == {"llama2_70b_bf16_gqa", "cow_parallel_sampling_f16",
                                        "llama2_7b_fp8_long"}


def test_every_ncu_traffic_figure_is_in_its_profile():
    """Each DRAM-traffic constant bench.py reports names a tracked summary
    under profiles/ that prints both byte counts and the source hash the
    constant is valid for."""
    import os
    import re
    tables = [bench.NCU_TRAFFIC, bench.NCU_PREFILL_TRAFFIC, bench.NCU_HASH_TRAFFIC]
    for table in tables:
        for name, tr in table.items():
            path = os.path.join(bench.ROOT, tr["profile"])
            assert os.path.exists(path), (name, path)
            text = open(path).read().replace(",", "")
            assert tr["src_sha"] in text, (name, "source hash missing")
            # the constant is read + write from the capture, both printed
            counts = [int(x) for x in re.findall(r"(\d+) B\b", text)]
            found = any(a + b == tr["bytes_per_launch"] for a in counts for b in counts)
            assert found, (name, "byte counts missing")
    # (when the sources change after a capture, bench.py reports the traffic
    # as null until it is captured again)
