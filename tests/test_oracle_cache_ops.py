"""Pins of the oracle's kv_append and copy_blocks byte models.

* append with matching types is a scatter: the cache viewed as
  [block, slot, head, d] and flattened over (block, slot) is indexed by the slot
  number (numpy fancy indexing);
* an E4M3 append stores the E4M3 code of fp32(x) * fp32(1/scale) (the encoder is
  pinned in test_oracle_elements.py; the multiply is checked in float32 here);
* untouched slots keep their sentinel bytes; a negative slot writes nothing;
  slots outside the pool are skipped and counted;
* copy_blocks gives every dst block the src block's bytes, per layer, and leaves
  every other byte alone.
"""
import numpy as np
import pytest
import torch

import oracle

SENTINEL16 = 0xA5A5
SENTINEL8 = 0xA5


def _scatter_ref(cache, rows, slots):
    nb, hkv, bs, d = cache.shape
    view = cache.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d).copy()
    keep = slots >= 0
    view[slots[keep]] = rows[keep]
    return view.reshape(nb, bs, hkv, d).transpose(0, 2, 1, 3)


@pytest.mark.parametrize("code", [oracle.F16, oracle.BF16])
def test_append_same_type_is_a_scatter(code):
    rng = np.random.default_rng(21)
    nb, hkv, bs, d, T = 9, 3, 4, 8, 17
    kc = np.full((nb, hkv, bs, d), SENTINEL16, np.uint16)
    vc = np.full((nb, hkv, bs, d), SENTINEL16, np.uint16)
    slots = rng.choice(nb * bs, T, replace=False).astype(np.int64)
    slots[[2, 7]] = -1
    k = rng.integers(0, 1 << 16, (T, hkv, d), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, (T, hkv, d), dtype=np.uint16)
    kref, vref = _scatter_ref(kc, k, slots), _scatter_ref(vc, v, slots)
    assert oracle.kv_append(kc, vc, code, k, v, code, slots) == 0
    assert np.array_equal(kc, kref) and np.array_equal(vc, vref)
    assert (kc == SENTINEL16).sum() == kc.size - (T - 2) * hkv * d


def test_append_e4m3_quantises_with_fp32_reciprocal():
    rng = np.random.default_rng(22)
    nb, hkv, bs, d, T = 6, 2, 8, 16, 20
    kc = np.full((nb, hkv, bs, d), SENTINEL8, np.uint8)
    vc = np.full((nb, hkv, bs, d), SENTINEL8, np.uint8)
    slots = rng.choice(nb * bs, T, replace=False).astype(np.int64)
    kf = (rng.standard_normal((T, hkv, d)) * 3).astype(np.float32)
    vf = (rng.standard_normal((T, hkv, d)) * 3).astype(np.float32)
    kb = torch.from_numpy(kf).to(torch.bfloat16)
    vb = torch.from_numpy(vf).to(torch.bfloat16)
    k_scale, v_scale = np.float32(0.021), np.float32(0.0077)   # v saturates
    oracle.kv_append(kc, vc, oracle.E4M3, kb.view(torch.int16).numpy().view(np.uint16),
                     vb.view(torch.int16).numpy().view(np.uint16), oracle.BF16, slots,
                     k_scale=float(k_scale), v_scale=float(v_scale))
    yk = kb.float().numpy() * (np.float32(1) / k_scale)            # fp32 multiply
    yv = vb.float().numpy() * (np.float32(1) / v_scale)
    assert yk.dtype == np.float32 and np.abs(yv).max() > 448
    kref = _scatter_ref(np.full_like(kc, SENTINEL8), oracle.encode_e4m3(yk), slots)
    vref = _scatter_ref(np.full_like(vc, SENTINEL8), oracle.encode_e4m3(yv), slots)
    assert np.array_equal(kc, kref) and np.array_equal(vc, vref)
    # away from saturation the stored code is torch's own fp8 cast of the product
    ok = np.abs(yk) < 448
    tk = torch.from_numpy(yk).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.encode_e4m3(yk)[ok], tk[ok])


def test_append_skips_and_counts_out_of_pool_slots():
    nb, hkv, bs, d = 2, 1, 4, 8
    kc = np.full((nb, hkv, bs, d), SENTINEL16, np.uint16)
    vc = kc.copy()
    k = np.ones((3, hkv, d), np.uint16)
    n = oracle.kv_append(kc, vc, oracle.F16, k, k, oracle.F16,
                         np.array([nb * bs, 10 ** 9, 3], np.int64))
    assert n == 2
    assert (kc != SENTINEL16).sum() == d and np.all(kc[0, 0, 3] == 1)


def test_append_rejects_unsupported_pairing():
    kc = np.zeros((1, 1, 4, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.kv_append(kc, kc.copy(), oracle.BF16, np.zeros((1, 1, 8), np.uint16),
                         np.zeros((1, 1, 8), np.uint16), oracle.F16, np.array([0]))


def test_copy_blocks_copies_whole_blocks_every_layer():
    rng = np.random.default_rng(23)
    layers, nb, hkv, bs, d = 3, 12, 2, 4, 8
    ks = [rng.integers(0, 1 << 16, (nb, hkv, bs, d), dtype=np.uint16) for _ in range(layers)]
    vs = [rng.integers(0, 1 << 16, (nb, hkv, bs, d), dtype=np.uint16) for _ in range(layers)]
    before_k = [k.copy() for k in ks]
    before_v = [v.copy() for v in vs]
    pairs = np.array([[1, 7], [1, 8], [4, 0], [11, 2]], np.int64)
    oracle.copy_blocks(ks, vs, pairs)
    for l in range(layers):
        ek, ev = before_k[l].copy(), before_v[l].copy()
        for src, dst in pairs:
            ek[dst] = before_k[l][src]
            ev[dst] = before_v[l][src]
        assert np.array_equal(ks[l], ek) and np.array_equal(vs[l], ev)


def test_copy_blocks_uses_the_state_before_the_call():
    # a dst that is also a later src: the later copy reads the original bytes
    nb = 4
    k = np.arange(nb * 8, dtype=np.uint16).reshape(nb, 1, 2, 4)
    v = k.copy()
    orig = k.copy()
    oracle.copy_blocks([k], [v], np.array([[0, 1], [1, 2]], np.int64))
    assert np.array_equal(k[1], orig[0]) and np.array_equal(k[2], orig[1])


def test_copy_blocks_rejects_out_of_pool_pairs_without_writing():
    k = np.zeros((3, 1, 2, 4), np.uint16)
    v = k.copy()
    k[0] = 7
    with pytest.raises(IndexError):
        oracle.copy_blocks([k], [v], np.array([[0, 1], [0, 3]], np.int64))
    assert np.all(k[1] == 0)
    oracle.copy_blocks([k], [v], np.zeros((0, 2), np.int64))
