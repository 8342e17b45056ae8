"""Parity of the CUDA path (through the C ABI) with the oracle, on the same
seeded inputs, at sizes the oracle finishes in seconds.

* kv_append and copy_blocks: the whole K and V caches, byte for byte,
  including the untouched sentinel bytes;
* decode attention: |gpu - oracle| <= 2e-3 + 2e-3 |oracle| elementwise.
"""
import numpy as np
import pytest
import torch

import harness as H
import oracle
from paged_kv_cache_130_gb300 import binding as B
from paged_kv_cache_130_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    H.build_library()


SMALL = {
    "tiny_f16": lambda: W.tiny_f16(),
    "opt13b_f16": lambda: W.opt13b_f16(num_seqs=6),
    "llama2_70b_bf16_gqa": lambda: W.llama2_70b_bf16_gqa(num_seqs=3),
    "cow_parallel_sampling_f16": lambda: W.cow_parallel_sampling_f16(num_prompts=2),
    "llama2_7b_fp8_long": lambda: W.llama2_7b_fp8_long(num_seqs=2),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_workload_end_to_end(name):
    w = SMALL[name]()
    g = H.GpuRun(w)
    o = H.OracleRun(w)
    # prefill
    g.prefill()
    o.prefill()
    torch.cuda.synchronize()
    assert np.array_equal(H.to_bits(g.k_cache), o.k_cache), "prefill K bytes"
    assert np.array_equal(H.to_bits(g.v_cache), o.v_cache), "prefill V bytes"
    # copy-on-write copies, then the step's append
    g.copy()
    o.copy()
    g.step()
    o.step()
    torch.cuda.synchronize()
    assert np.array_equal(H.to_bits(g.k_cache), o.k_cache), "step K bytes"
    assert np.array_equal(H.to_bits(g.v_cache), o.v_cache), "step V bytes"
    # decode
    out = g.decode()
    ref = o.decode()
    torch.cuda.synchronize()
    H.assert_attention_close(H.out_to_double(out), ref, name, w.io_dtype)
    assert int(g.dev_err.item()) == 0


def _random_problem(rng, cache_dt, q_dt, D, BS, G, Hkv, ctx, nb_extra=7):
    """A direct-built problem (not a named workload) for shape sweeps."""
    S = len(ctx)
    nblk = [-(-c // BS) for c in ctx]
    nb = sum(nblk) + nb_extra
    order = rng.permutation(nb)
    mb = max(max(nblk), 1)
    bt = np.full((S, mb), -1, np.int32)
    pos = 0
    for s in range(S):
        for i in range(nblk[s]):
            bt[s, i] = order[pos]
            pos += 1
    shape = (nb, Hkv, BS, D)
    if cache_dt == W.E4M3:
        kc = rng.integers(0, 256, shape, dtype=np.uint8)
        vc = rng.integers(0, 256, shape, dtype=np.uint8)
        # no NaN codes inside the used slots
        kc[(kc & 0x7f) == 0x7f] = 0x7e
        vc[(vc & 0x7f) == 0x7f] = 0x3f
    else:
        kc = W._to_bits(rng.standard_normal(shape, dtype=np.float32), cache_dt)
        vc = W._to_bits(rng.standard_normal(shape, dtype=np.float32), cache_dt)
    # unused slots of the last block of each sequence hold NaN
    for s in range(S):
        if ctx[s] % BS:
            b = bt[s, nblk[s] - 1]
            kc.view(np.uint8).reshape(nb, Hkv, BS, -1)[b, :, ctx[s] % BS:, :] = 0xFF
            vc.view(np.uint8).reshape(nb, Hkv, BS, -1)[b, :, ctx[s] % BS:, :] = 0xFF
    q = W._to_bits(rng.standard_normal((S, G * Hkv, D), dtype=np.float32), q_dt)
    ctx = np.asarray(ctx, np.int32)
    return kc, vc, q, bt, ctx


def _gpu_decode(kc, vc, cache_dt, q, q_dt, bt, ctx, scale, k_scale=1.0, v_scale=1.0,
                partition_size=0, max_ctx=None):
    kt = H.to_device(kc, cache_dt)
    vt = H.to_device(vc, cache_dt)
    desc = B.cache_desc(kt, vt, k_scale, v_scale)
    qt = H.to_device(q, q_dt)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = B.pkv_paged_attention_decode(
        desc, qt, torch.from_numpy(bt).cuda(), torch.from_numpy(ctx).cuda(),
        int(ctx.max()) if max_ctx is None else max_ctx, scale,
        partition_size=partition_size, dev_err=err)
    torch.cuda.synchronize()
    return out, int(err.item()), (kt, vt, desc)


SHAPES = []
for cdt, qdt in ((W.F16, W.F16), (W.BF16, W.BF16), (W.E4M3, W.F16), (W.E4M3, W.BF16)):
    for D in (64, 128):
        for BS in (8, 16, 32):
            for G in (1, 2, 8, 16):
                SHAPES.append((cdt, qdt, D, BS, G))


@pytest.mark.parametrize("cdt,qdt,D,BS,G", SHAPES)
def test_decode_shapes(cdt, qdt, D, BS, G):
    rng = np.random.default_rng(1000 + D + BS + 7 * G + 31 * cdt + 97 * qdt)
    Hkv = 2
    ctx = [1, BS - 1, BS, BS + 1, 3 * BS + 5, 70, 200]
    kc, vc, q, bt, ctxa = _random_problem(rng, cdt, qdt, D, BS, G, Hkv, ctx)
    ks, vs = (0.03, 0.02) if cdt == W.E4M3 else (1.0, 1.0)
    scale = float(np.float32(1 / np.sqrt(D)))
    for ps in (0, 2 * BS):
        out, err, _ = _gpu_decode(kc, vc, cdt, q, qdt, bt, ctxa, scale, ks, vs, partition_size=ps)
        ref = oracle.paged_attention_decode(kc, vc, cdt, q, qdt, bt, ctxa, scale, ks, vs)
        H.assert_attention_close(H.out_to_double(out), ref,
                                 "shape %s partition %d" % ((cdt, qdt, D, BS, G), ps), qdt)
        assert err == 0


@pytest.mark.parametrize("cdt,qdt,G", [(W.F16, W.F16, 1), (W.BF16, W.BF16, 8),
                                        (W.E4M3, W.BF16, 1)])
def test_large_batch(cdt, qdt, G):
    """More sequences than the kernels rank by length (128) and than the
    streaming kernel keeps context lengths for in shared memory (512): the
    unsorted walk and the lengths read from global memory."""
    rng = np.random.default_rng(2024 + G + 5 * cdt)
    BS, D, Hkv = 16, 128, 2
    ctx = list(rng.integers(1, 120, size=600))
    ctx[3] = 0
    ctx[599] = 1
    ctx[77] = 400
    kc, vc, q, bt, ctxa = _random_problem(rng, cdt, qdt, D, BS, G, Hkv, ctx)
    ks, vs = (0.03, 0.02) if cdt == W.E4M3 else (1.0, 1.0)
    scale = float(np.float32(1 / np.sqrt(D)))
    ref = oracle.paged_attention_decode(kc, vc, cdt, q, qdt, bt, ctxa, scale, ks, vs)
    for ps in (0, 4 * BS):
        out, err, _ = _gpu_decode(kc, vc, cdt, q, qdt, bt, ctxa, scale, ks, vs, partition_size=ps)
        H.assert_attention_close(H.out_to_double(out), ref,
                                 "600 sequences %s partition %d" % ((cdt, qdt, G), ps), qdt)
        assert err == 0


@pytest.mark.parametrize("cdt,G", [(W.F16, 1), (W.BF16, 1), (W.F16, 8), (W.BF16, 8),
                                    (W.E4M3, 1)])
def test_single_token_context_returns_v_exactly(cdt, G):
    rng = np.random.default_rng(7)
    qdt = W.BF16 if cdt == W.E4M3 else cdt
    kc, vc, q, bt, ctx = _random_problem(rng, cdt, qdt, 128, 16, G, 2, [1, 1, 1])
    out, err, _ = _gpu_decode(kc, vc, cdt, q, qdt, bt, ctx, 0.1)
    ref = oracle.paged_attention_decode(kc, vc, cdt, q, qdt, bt, ctx, 0.1)
    got = H.out_to_double(out)
    if cdt == W.E4M3:
        # every E4M3 value is exact in bf16: the weight is exactly 1
        assert np.array_equal(got, ref)
    else:
        assert np.array_equal(got, ref)
    assert err == 0


def test_e4m3_decode_table_through_the_kernel():
    """All 256 codes as the V of a one-token context: out = decoded value."""
    codes = np.arange(256, dtype=np.uint8)
    D, BS = 128, 16
    kc = np.zeros((2, 1, BS, D), np.uint8)
    vc = np.zeros((2, 1, BS, D), np.uint8)
    vc[0, 0, 0, :] = codes[:128]
    vc[1, 0, 0, :] = codes[128:]
    q = np.zeros((2, 1, D), np.uint16)
    bt = np.array([[0], [1]], np.int32)
    ctx = np.array([1, 1], np.int32)
    out, err, _ = _gpu_decode(kc, vc, W.E4M3, q, W.BF16, bt, ctx, 1.0)
    got = H.out_to_double(out).reshape(-1)
    ref = oracle.decode(oracle.E4M3, codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    # equal values (the sign of a zero output is not defined by the sum)
    assert np.array_equal(got[~nan], ref[~nan])


def test_empty_context_gives_zero_and_padding_is_ignored():
    rng = np.random.default_rng(8)
    kc, vc, q, bt, ctx = _random_problem(rng, W.F16, W.F16, 64, 16, 1, 2, [0, 5, 0])
    bt[0, :] = 10 ** 6          # never read: context 0
    out, err, _ = _gpu_decode(kc, vc, W.F16, q, W.F16, bt, ctx, 0.2, max_ctx=64)
    got = H.out_to_double(out)
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    ref = oracle.paged_attention_decode(kc, vc, W.F16, q[1:2], W.F16, bt[1:2], ctx[1:2], 0.2)
    H.assert_attention_close(got[1:2], ref, "empty neighbours")
    assert err == 0


@pytest.mark.parametrize("G,cdt", [(1, W.F16), (8, W.BF16), (1, W.E4M3)])
def test_partition_boundaries(G, cdt):
    rng = np.random.default_rng(9)
    BS, P = 16, 64
    qdt = W.BF16 if cdt != W.F16 else W.F16
    ctx = [P - 1, P, P + 1, 2 * P, 2 * P + 1, 5 * P + 3, 1, 17]
    kc, vc, q, bt, ctxa = _random_problem(rng, cdt, qdt, 128, BS, G, 2, ctx)
    ks, vs = (0.05, 0.04) if cdt == W.E4M3 else (1.0, 1.0)
    out, err, _ = _gpu_decode(kc, vc, cdt, q, qdt, bt, ctxa, 0.09, ks, vs, partition_size=P)
    ref = oracle.paged_attention_decode(kc, vc, cdt, q, qdt, bt, ctxa, 0.09, ks, vs)
    H.assert_attention_close(H.out_to_double(out), ref, "partitions", qdt)
    assert err == 0


# (partition size, contexts): units of four 32-token partitions, and of two
# 1024-token partitions
SCHEDULE_CASES = [(32, [1, 17, 31, 32, 8 * 32, 8 * 32 + 1, 13 * 32 + 5, 20 * 32 + 3, 31 * 32,
                        40 * 32 + 7]),
                  (1024, [9000, 8193, 5000, 1500, 300])]


@pytest.mark.parametrize("case", [0, 1])
@pytest.mark.parametrize("cdt", [W.F16, W.E4M3])
def test_claim_schedules_agree_bit_for_bit(cdt, case):
    """The streaming kernel hands out its work by one of two schedules: the
    compact one (the batch ranked longest first, units where a sequence has
    no partition left skipped, the last partitions handed out one at a time)
    or the plain one (partition blocks x sequences x heads), taken when the
    lengths do not rank in partition order, as with a context past
    max_context_len.  A partition's result does not depend on which CTA took
    it or when, so the rows both batches share come out the same, bit for
    bit; the compact one is checked against the oracle too."""
    rng = np.random.default_rng(31 + cdt + 7 * case)
    BS, D, G, Hkv = 16, 128, 1, 2
    # at least eight partitions in the longest context: claimed
    # min(4, 2048 / P) partitions at a time
    P, ctx = SCHEDULE_CASES[case]
    qdt = W.F16 if cdt == W.F16 else W.BF16
    kc, vc, q, bt, ctxa = _random_problem(rng, cdt, qdt, D, BS, G, Hkv, ctx)
    ks, vs = (0.05, 0.04) if cdt == W.E4M3 else (1.0, 1.0)
    max_ctx = int(ctxa.max())
    out1, err1, _ = _gpu_decode(kc, vc, cdt, q, qdt, bt, ctxa, 0.09, ks, vs, partition_size=P)
    ref = oracle.paged_attention_decode(kc, vc, cdt, q, qdt, bt, ctxa, 0.09, ks, vs)
    H.assert_attention_close(H.out_to_double(out1), ref, "compact schedule", qdt)
    assert err1 == 0
    # the same batch and one more sequence whose context is past
    # max_context_len: it ranks first with one (zero) item, so the lengths no
    # longer rank in partition order and the plain schedule runs
    bt2 = np.vstack([bt, bt[:1]])
    ctx2 = np.append(ctxa, np.int32(max_ctx + 5)).astype(np.int32)
    q2 = np.concatenate([q, q[:1]])
    out2, err2, _ = _gpu_decode(kc, vc, cdt, q2, qdt, bt2, ctx2, 0.09, ks, vs, partition_size=P,
                                max_ctx=max_ctx)
    assert err2 & B.PKV_DEVERR_CONTEXT
    assert torch.all(out2[-1] == 0)
    assert torch.equal(out2[:-1].view(torch.int16), out1.view(torch.int16))


@pytest.mark.parametrize("cdt", [W.F16, W.E4M3])
def test_schedule_with_hundreds_of_partitions(cdt):
    """Partitions of one block over contexts of up to 600 blocks: more
    schedule entries than the compact schedule keeps, so the plain one runs;
    and a batch whose work is too small for a tail of full units, handed out
    one partition at a time."""
    rng = np.random.default_rng(37 + cdt)
    BS, D, G, Hkv = 16, 128, 1, 2
    qdt = W.F16 if cdt == W.F16 else W.BF16
    ks, vs = (0.05, 0.04) if cdt == W.E4M3 else (1.0, 1.0)
    for ctx in ([600 * BS, 5000, 33, 1], [9 * BS, 1, 2]):
        kc, vc, q, bt, ctxa = _random_problem(rng, cdt, qdt, D, BS, G, Hkv, ctx)
        out, err, _ = _gpu_decode(kc, vc, cdt, q, qdt, bt, ctxa, 0.09, ks, vs,
                                  partition_size=BS)
        ref = oracle.paged_attention_decode(kc, vc, cdt, q, qdt, bt, ctxa, 0.09, ks, vs)
        H.assert_attention_close(H.out_to_double(out), ref, "contexts %s" % ctx, qdt)
        assert err == 0


@pytest.mark.parametrize("G", [1, 8])
def test_placement_does_not_change_a_bit(G):
    """The kernels' reduction order does not depend on physical block ids."""
    rng = np.random.default_rng(10)
    BS = 16
    ctx = [37, 300, 129]
    kc, vc, q, bt, ctxa = _random_problem(rng, W.BF16, W.BF16, 128, BS, G, 2, ctx)
    out1, _, _ = _gpu_decode(kc, vc, W.BF16, q, W.BF16, bt, ctxa, 0.1, partition_size=64)
    # move every used block to a new physical place
    nb = kc.shape[0]
    perm = rng.permutation(nb)
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(bt >= 0, perm[np.clip(bt, 0, None)], -1).astype(np.int32)
    out2, _, _ = _gpu_decode(kc2, vc2, W.BF16, q, W.BF16, bt2, ctxa, 0.1, partition_size=64)
    assert torch.equal(out1, out2)


@pytest.mark.parametrize("name", ["opt13b_f16", "llama2_7b_fp8_long"])
def test_repeated_decode_is_bit_identical(name):
    """Work items go to CTAs in whatever order the device counter hands them
    out, so the warp that holds a block residue changes from run to run; the
    result must not."""
    w = W.opt13b_f16(num_seqs=48) if name == "opt13b_f16" else W.llama2_7b_fp8_long(num_seqs=6)
    g = H.GpuRun(w)
    g.prefill()
    g.step()
    first = g.decode().clone()
    for i in range(8):
        # a decode of another batch size in between moves the counters' timing
        if i % 2:
            g.decode(partition_size=w.block_size * 4)
        out = g.decode()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), first.view(torch.int16)), "run %d" % i
    assert int(g.dev_err.item()) == 0


def test_lse_reduce_merges_oracle_partials():
    """The reduce kernel alone, fed partials the oracle computed per range:
    rows of 2 to 7 partials (one load round), 10 and 35 (partials' m and l
    kept in registers) and 132 (past what the registers keep)."""
    rng = np.random.default_rng(11)
    BS, P, D, Hkv = 16, 32, 128, 2
    ctx = [33, 64, 65, 200, 31, 300, 1100, 4200]
    kc, vc, q, bt, ctxa = _random_problem(rng, W.F16, W.F16, D, BS, 1, Hkv, ctx)
    S, Hq = len(ctx), Hkv
    maxp = -(-int(ctxa.max()) // P)
    m = np.full((S, Hq, maxp), -np.inf, np.float32)
    l = np.zeros((S, Hq, maxp), np.float32)
    o = np.zeros((S, Hq, maxp, D), np.float32)
    scale = 0.11
    for p in range(maxp):
        op, mp, lp = oracle.attention_range(kc, vc, W.F16, q, W.F16, bt, ctxa, scale,
                                            p * P, (p + 1) * P)
        m[:, :, p] = mp * np.log2(np.e)
        l[:, :, p] = lp
        o[:, :, p, :] = op
    rows = S * Hq * maxp
    ml = -(-4 * rows // 256) * 256
    ws = np.zeros(2 * ml + -(-4 * rows * D // 256) * 256, np.uint8)
    ws[:4 * rows].view(np.float32)[:] = m.reshape(-1)
    ws[ml:ml + 4 * rows].view(np.float32)[:] = l.reshape(-1)
    ws[2 * ml:2 * ml + 4 * rows * D].view(np.float32)[:] = o.reshape(-1)
    wst = torch.from_numpy(ws).cuda()
    out = torch.zeros((S, Hq, D), dtype=torch.float16, device="cuda")
    B.pkv_lse_reduce(S, Hq, D, torch.from_numpy(ctxa).cuda(), int(ctxa.max()), P, wst, out)
    torch.cuda.synchronize()
    ref = oracle.paged_attention_decode(kc, vc, W.F16, q, W.F16, bt, ctxa, scale)
    got = H.out_to_double(out)
    multi = np.array([c > P for c in ctx])
    H.assert_attention_close(got[multi], ref[multi], "reduce")
    assert np.all(got[~multi] == 0)      # single-partition rows are left alone


def test_copy_blocks_multi_layer_bit_exact():
    rng = np.random.default_rng(12)
    layers, nb, hkv, bs, d = 3, 40, 4, 16, 128
    ks = [rng.integers(0, 1 << 16, (nb, hkv, bs, d), dtype=np.uint16) for _ in range(layers)]
    vs = [rng.integers(0, 1 << 16, (nb, hkv, bs, d), dtype=np.uint16) for _ in range(layers)]
    pairs = np.array([[3, 30], [3, 31], [7, 0], [39, 12], [5, 6]], np.int64)
    kt = [H.to_device(k, W.F16) for k in ks]
    vt = [H.to_device(v, W.F16) for v in vs]
    descs = [B.cache_desc(a, b) for a, b in zip(kt, vt)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.pkv_copy_blocks(descs, torch.from_numpy(pairs).cuda(), dev_err=err)
    torch.cuda.synchronize()
    oracle.copy_blocks(ks, vs, pairs)
    for l in range(layers):
        assert np.array_equal(H.to_bits(kt[l]), ks[l])
        assert np.array_equal(H.to_bits(vt[l]), vs[l])
    assert int(err.item()) == 0


def test_device_range_checks_skip_and_flag():
    """Out-of-range indices are caught by the kernels' own checks: the access
    is skipped and a bit is set; nothing outside the buffers is touched."""
    rng = np.random.default_rng(13)
    BS, D = 16, 64
    nb = 8
    kc = W._to_bits(rng.standard_normal((nb, 1, BS, D), dtype=np.float32), W.F16)
    vc = W._to_bits(rng.standard_normal((nb, 1, BS, D), dtype=np.float32), W.F16)
    kt, vt = H.to_device(kc, W.F16), H.to_device(vc, W.F16)
    desc = B.cache_desc(kt, vt)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # append: one slot past the pool, one far past it, one valid
    k = H.to_device(np.zeros((3, 1, D), np.uint16), W.F16)
    slots = torch.tensor([nb * BS, 10 ** 12, 5], dtype=torch.int64, device="cuda")
    B.pkv_kv_append(desc, k, k, slots, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == B.PKV_DEVERR_SLOT
    after = H.to_bits(kt)
    expect = kc.copy()
    expect[0, 0, 5, :] = 0
    assert np.array_equal(after, expect)
    # copy: a pair past the pool
    err.zero_()
    B.pkv_copy_blocks(desc, torch.tensor([[0, nb], [nb + 5, 1]], dtype=torch.int64,
                                         device="cuda"), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == B.PKV_DEVERR_COPY_PAIR
    assert np.array_equal(H.to_bits(kt), expect)
    # decode: a block id past the pool, a context past the table
    err.zero_()
    q = H.to_device(W._to_bits(rng.standard_normal((2, 1, D), dtype=np.float32), W.F16), W.F16)
    bt = torch.tensor([[0, nb + 3], [1, 2]], dtype=torch.int32, device="cuda")
    cl = torch.tensor([20, 40], dtype=torch.int32, device="cuda")
    out = B.pkv_paged_attention_decode(desc, q, bt, cl, 40, 0.1, dev_err=err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & B.PKV_DEVERR_BLOCK_ID and e & B.PKV_DEVERR_CONTEXT
    assert torch.all(out[1] == 0)
    assert torch.isfinite(out).all()
