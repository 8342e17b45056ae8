"""Pins of the oracle's block swap (device pool <-> host pool).

* round trip: swapping blocks out and back into other blocks reproduces their
  bytes, and every block no pair names keeps its sentinel;
* per-layer independence: each layer moves its own block, K and V alike;
* a pair outside either pool is refused.
"""
import numpy as np
import pytest

import oracle


def _pools(rng, layers, nb, shape=(2, 4, 8)):
    k = [rng.integers(0, 2 ** 16, size=(nb,) + shape, dtype=np.uint16) for _ in range(layers)]
    v = [rng.integers(0, 2 ** 16, size=(nb,) + shape, dtype=np.uint16) for _ in range(layers)]
    return k, v


def test_round_trip_restores_bytes():
    rng = np.random.default_rng(1)
    dk, dv = _pools(rng, 3, 20)
    hk = [np.full((6,) + a.shape[1:], 0xA5A5, np.uint16) for a in dk]
    hv = [np.full((6,) + a.shape[1:], 0xA5A5, np.uint16) for a in dv]
    out_pairs = np.array([[4, 0], [17, 3], [9, 5]])
    oracle.swap_blocks(dk, dv, hk, hv, out_pairs)
    for l in range(3):
        assert np.array_equal(hk[l][[0, 3, 5]], dk[l][[4, 17, 9]])
        assert np.array_equal(hv[l][[0, 3, 5]], dv[l][[4, 17, 9]])
        assert np.all(hk[l][[1, 2, 4]] == 0xA5A5) and np.all(hv[l][[1, 2, 4]] == 0xA5A5)
    before = [a.copy() for a in dk]
    back = np.array([[0, 1], [3, 2], [5, 19]])       # into other device blocks
    oracle.swap_blocks(hk, hv, dk, dv, back)
    for l in range(3):
        assert np.array_equal(dk[l][[1, 2, 19]], before[l][[4, 17, 9]])
        untouched = [b for b in range(20) if b not in (1, 2, 19)]
        assert np.array_equal(dk[l][untouched], before[l][untouched])


def test_pairs_outside_a_pool_are_refused():
    rng = np.random.default_rng(2)
    dk, dv = _pools(rng, 1, 4)
    hk, hv = _pools(rng, 1, 2)
    with pytest.raises(IndexError):
        oracle.swap_blocks(dk, dv, hk, hv, [[1, 2]])
    with pytest.raises(IndexError):
        oracle.swap_blocks(dk, dv, hk, hv, [[-1, 0]])
