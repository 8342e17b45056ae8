"""Pins of the oracle's causal prefill attention over the paged cache.

* library routine: a dense causal softmax attention in numpy over the
  contiguous [ctx, D] K/V (the layout paging replaces), with the new queries
  at the last positions of each context, equals the paged prefill for any
  block placement, with grouped heads and a context cached before the new
  tokens (chunked prefill);
* causality: changing the K/V of tokens after a query's position leaves its
  output bit-identical, changing one at or before it does not;
* closed form: the first token of a prompt with no earlier context returns its
  own V exactly.
"""
import numpy as np
import pytest

import oracle

F16, BF16 = 0, 1


def _bits(x, code):
    if code == F16:
        return x.astype(np.float16).view(np.uint16)
    # bf16: round-to-nearest-even of the fp32 bits
    u = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _vals(bits, code):
    if code == F16:
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _problem(rng, code, ctx, new, hkv, g, d, bs):
    """Caches holding every sequence's context at a random placement, the
    contiguous copies of the same K/V, and the new tokens' queries."""
    nseq = len(ctx)
    nblk = [(c + bs - 1) // bs for c in ctx]
    nb = sum(nblk) + 3
    perm = rng.permutation(nb)
    tables = np.full((nseq, max(nblk)), -1, np.int32)
    k_cache = np.zeros((nb, hkv, bs, d), np.uint16)
    v_cache = np.zeros((nb, hkv, bs, d), np.uint16)
    dense_k, dense_v = [], []
    used = 0
    for s in range(nseq):
        tables[s, :nblk[s]] = perm[used:used + nblk[s]]
        used += nblk[s]
        k = _bits(rng.standard_normal((ctx[s], hkv, d)), code)
        v = _bits(rng.standard_normal((ctx[s], hkv, d)), code)
        slots = np.array([tables[s, t // bs] * bs + t % bs for t in range(ctx[s])], np.int64)
        oracle.kv_append(k_cache, v_cache, code, k, v, code, slots)
        dense_k.append(_vals(k, code))
        dense_v.append(_vals(v, code))
    cu = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    q = _bits(rng.standard_normal((int(cu[-1]), hkv * g, d)), code)
    return k_cache, v_cache, tables, cu, q, dense_k, dense_v


def _dense_causal(q_vals, cu, ctx, dense_k, dense_v, g, scale):
    out = np.zeros(q_vals.shape)
    for s in range(len(ctx)):
        n = cu[s + 1] - cu[s]
        for j in range(n):
            p = ctx[s] - n + j
            for h in range(q_vals.shape[1]):
                kk = dense_k[s][:p + 1, h // g, :]
                vv = dense_v[s][:p + 1, h // g, :]
                x = scale * (kk @ q_vals[cu[s] + j, h])
                w = np.exp(x - x.max())
                out[cu[s] + j, h] = (w @ vv) / w.sum()
    return out


@pytest.mark.parametrize("code,hkv,g,d,bs", [(F16, 2, 1, 16, 4), (BF16, 2, 3, 8, 8),
                                             (F16, 1, 4, 32, 16)])
def test_prefill_equals_dense_causal_attention(code, hkv, g, d, bs):
    rng = np.random.default_rng(11 + g)
    ctx = [7, 40, 33, 1]
    new = [7, 12, 5, 1]           # whole prompt, chunk after 28 cached, after 28, single
    kc, vc, bt, cu, q, dk, dv = _problem(rng, code, ctx, new, hkv, g, d, bs)
    scale = 0.3
    got = oracle.paged_attention_prefill(kc, vc, code, q, code, cu, bt, ctx, scale)
    want = _dense_causal(_vals(q, code), cu, ctx, dk, dv, g, float(np.float32(scale)))
    assert np.max(np.abs(got - want)) < 1e-12


def test_prefill_is_causal():
    rng = np.random.default_rng(3)
    ctx, new = [30], [10]
    kc, vc, bt, cu, q, _, _ = _problem(rng, F16, ctx, new, 1, 2, 16, 4)
    base = oracle.paged_attention_prefill(kc, vc, F16, q, F16, cu, bt, ctx, 0.25)
    # token 25 is after the positions of rows 0..4 (20..24) and not after 5..9
    blk, off = bt[0, 25 // 4], 25 % 4
    kc2 = kc.copy()
    kc2[blk, 0, off, :] = _bits(np.full(16, 3.0), F16)
    moved = oracle.paged_attention_prefill(kc2, vc, F16, q, F16, cu, bt, ctx, 0.25)
    assert np.array_equal(moved[:5], base[:5])
    assert np.all(np.any(moved[5:] != base[5:], axis=2))


def test_first_prompt_token_returns_its_v():
    rng = np.random.default_rng(4)
    ctx, new = [9], [9]
    kc, vc, bt, cu, q, _, dv = _problem(rng, BF16, ctx, new, 2, 2, 8, 4)
    out = oracle.paged_attention_prefill(kc, vc, BF16, q, BF16, cu, bt, ctx, 0.5)
    for h in range(4):
        assert np.array_equal(out[0, h], dv[0][0, h // 2])
