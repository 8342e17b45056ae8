"""Pins of the oracle's decode attention.

* brute force: tiny problems in pure Python (math.fsum / math.exp);
* library routine: numpy softmax attention over a contiguous [ctx, D] layout
  (the layout paging replaces) equals the paged result for any placement;
* permutation invariance: the physical placement of blocks does not change a bit;
* closed forms: a one-token context returns that token's V; equal keys or a zero
  query return the mean of V; two tokens give a sigmoid blend;
* grouped heads: a GQA problem equals the MHA problem with each KV head repeated
  for its group of consecutive query heads;
* partial ranges merge back into the whole by the log-sum-exp rule.
"""
import math

import numpy as np
import pytest

import oracle


def _problem(rng, S, H, Hkv, D, BS, ctx, nb=None, dtype=oracle.F16, sigma=1.0, perm=True):
    ctx = np.asarray(ctx, np.int32)
    nblk = [(-(-int(c) // BS)) for c in ctx]
    total = sum(nblk)
    nb = nb or total + 5
    # placement draws from its own stream so that values do not depend on it
    order = np.random.default_rng(999).permutation(nb) if perm else np.arange(nb)
    mb = max(nblk)
    bt = np.full((S, mb), -1, np.int32)
    k = np.zeros((nb, Hkv, BS, D), np.float32)
    v = np.zeros((nb, Hkv, BS, D), np.float32)
    dense_k, dense_v = [], []
    pos = 0
    for s in range(S):
        kk = (rng.standard_normal((ctx[s], Hkv, D)) * sigma).astype(np.float32)
        vv = (rng.standard_normal((ctx[s], Hkv, D)) * sigma).astype(np.float32)
        for i in range(nblk[s]):
            bt[s, i] = order[pos]
            pos += 1
        for t in range(ctx[s]):
            k[bt[s, t // BS], :, t % BS, :] = kk[t]
            v[bt[s, t // BS], :, t % BS, :] = vv[t]
        dense_k.append(kk)
        dense_v.append(vv)
    q = rng.standard_normal((S, H, D)).astype(np.float32)
    return dict(k=k, v=v, q=q, bt=bt, ctx=ctx, dense_k=dense_k, dense_v=dense_v)


def _bits16(x):
    return x.astype(np.float16).view(np.uint16)


def _run(p, scale, **kw):
    return oracle.paged_attention_decode(_bits16(p["k"]), _bits16(p["v"]), oracle.F16,
                                         _bits16(p["q"]), oracle.F16, p["bt"], p["ctx"],
                                         scale, **kw)


def _f16(x):
    return np.asarray(x, np.float32).astype(np.float16).astype(np.float64)


def test_brute_force_tiny():
    rng = np.random.default_rng(5)
    for ctx in ([1, 2, 3, 4], [4, 3, 2, 1]):
        for D in (1, 2, 4):
            p = _problem(rng, 4, 2, 2, D, 2, ctx)
            scale = float(np.float32(0.7))
            got = _run(p, scale)
            for s in range(4):
                for h in range(2):
                    qv = _f16(p["q"][s, h])
                    kk = _f16(p["dense_k"][s][:, h, :])
                    vv = _f16(p["dense_v"][s][:, h, :])
                    x = [scale * math.fsum(qv[d] * kk[t, d] for d in range(D))
                         for t in range(ctx[s])]
                    m = max(x)
                    w = [math.exp(xi - m) for xi in x]
                    den = math.fsum(w)
                    for d in range(D):
                        ref = math.fsum(w[t] * vv[t, d] for t in range(ctx[s])) / den
                        assert abs(got[s, h, d] - ref) <= 1e-14 * max(1.0, abs(ref))


def test_contiguous_layout_and_permutation_invariance():
    rng = np.random.default_rng(6)
    S, H, D, BS = 3, 4, 16, 4
    ctx = [13, 1, 29]
    p = _problem(np.random.default_rng(7), S, H, H, D, BS, ctx, nb=60, perm=True)
    p_id = _problem(np.random.default_rng(7), S, H, H, D, BS, ctx, nb=60, perm=False)
    scale = float(np.float32(1 / 4))
    a = _run(p, scale)
    b = _run(p_id, scale)
    assert np.array_equal(a, b)                              # bit-identical
    for s in range(S):
        for h in range(H):
            kk = _f16(p["dense_k"][s][:, h, :])
            vv = _f16(p["dense_v"][s][:, h, :])
            x = scale * (kk @ _f16(p["q"][s, h]))
            w = np.exp(x - x.max())
            ref = (w[:, None] * vv).sum(0) / w.sum()
            np.testing.assert_allclose(a[s, h], ref, rtol=1e-12, atol=1e-12)
    del rng


def test_closed_form_single_token_returns_v():
    p = _problem(np.random.default_rng(8), 2, 3, 3, 8, 4, [1, 1])
    got = _run(p, 0.3)
    for s in range(2):
        assert np.array_equal(got[s], _f16(p["dense_v"][s][0]))


def test_closed_form_equal_keys_or_zero_query_give_mean_v():
    rng = np.random.default_rng(9)
    p = _problem(rng, 2, 2, 2, 8, 4, [7, 12])
    for s in range(2):                     # all keys of a sequence equal
        for t in range(p["ctx"][s]):
            blk = p["bt"][s, t // 4]
            p["k"][blk, :, t % 4, :] = p["dense_k"][s][0]
    got = _run(p, 0.5)
    for s in range(2):
        np.testing.assert_allclose(got[s], _f16(p["dense_v"][s]).mean(0), rtol=0, atol=1e-15)
    p2 = _problem(np.random.default_rng(10), 2, 2, 2, 8, 4, [7, 12])
    p2["q"][:] = 0
    got2 = _run(p2, 0.5)
    for s in range(2):
        np.testing.assert_allclose(got2[s], _f16(p2["dense_v"][s]).mean(0), rtol=0, atol=1e-15)


def test_closed_form_two_tokens_sigmoid():
    p = _problem(np.random.default_rng(11), 1, 2, 2, 8, 4, [2])
    scale = float(np.float32(0.25))
    got = _run(p, scale)
    for h in range(2):
        qv = _f16(p["q"][0, h])
        k0, k1 = _f16(p["dense_k"][0][0, h]), _f16(p["dense_k"][0][1, h])
        v0, v1 = _f16(p["dense_v"][0][0, h]), _f16(p["dense_v"][0][1, h])
        sig = 1.0 / (1.0 + math.exp(-(scale * (qv @ k1) - scale * (qv @ k0))))
        np.testing.assert_allclose(got[0, h], sig * v1 + (1 - sig) * v0, rtol=1e-13, atol=1e-13)


def test_grouped_heads_equal_repeated_kv_heads():
    rng = np.random.default_rng(12)
    S, Hkv, G, D, BS = 2, 2, 3, 8, 4
    p = _problem(rng, S, Hkv * G, Hkv, D, BS, [9, 14])
    gqa = _run(p, 0.4)
    # expand: query head h reads KV head h // G (consecutive heads share)
    rep = dict(p)
    rep["k"] = np.repeat(p["k"], G, axis=1)
    rep["v"] = np.repeat(p["v"], G, axis=1)
    mha = _run(rep, 0.4)
    assert np.array_equal(gqa, mha)
    # and the grouping is not interleaved: head 1 differs from the result with KV head 1
    alt = dict(p)
    alt["k"] = np.tile(p["k"], (1, G, 1, 1))
    alt["v"] = np.tile(p["v"], (1, G, 1, 1))
    assert not np.array_equal(gqa, _run(alt, 0.4))


def test_scales_fold_into_logits_and_output():
    p = _problem(np.random.default_rng(13), 2, 2, 2, 8, 4, [6, 11])
    base = _run(p, 0.25)
    # V scale multiplies the output; K scale multiplies the logits
    got = _run(p, 0.25, v_scale=2.0)
    np.testing.assert_allclose(got, 2 * base, rtol=1e-15, atol=0)
    got = _run(p, 0.125, k_scale=2.0)
    np.testing.assert_allclose(got, base, rtol=1e-13, atol=1e-14)


def test_ranges_merge_to_whole():
    p = _problem(np.random.default_rng(14), 3, 2, 2, 8, 4, [1, 9, 30])
    whole = _run(p, 0.3)
    args = (_bits16(p["k"]), _bits16(p["v"]), oracle.F16, _bits16(p["q"]), oracle.F16,
            p["bt"], p["ctx"], 0.3)
    parts = [oracle.attention_range(*args, t0, t0 + 8) for t0 in range(0, 32, 8)]
    M = np.max([m for _, m, _ in parts], axis=0)
    num = sum(np.exp(m - M)[..., None] * o for o, m, _ in parts)
    den = sum(np.exp(m - M) * l for _, m, l in parts)
    np.testing.assert_allclose(num / den[..., None], whole, rtol=1e-13, atol=1e-14)
    o, m, l = parts[3]                       # tokens 24..31: only sequence 2 has any
    assert np.all(np.isneginf(m[:2])) and np.all(l[:2] == 0) and np.all(o[:2] == 0)


def test_bad_inputs_are_reported():
    p = _problem(np.random.default_rng(15), 1, 2, 2, 8, 4, [6])
    p["bt"][0, 1] = 10 ** 6
    with pytest.raises(ValueError):
        _run(p, 0.3)
    p = _problem(np.random.default_rng(15), 1, 3, 2, 8, 4, [6])
    with pytest.raises(ValueError):
        _run(p, 0.3)
