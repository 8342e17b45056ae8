"""Pins of the oracle's element conversions against the format definitions.

Each decoder is compared, code by code, with an independent library routine
(numpy's binary16, torch's bfloat16 and float8_e4m3fn casts) and with values
the formats fix.  The E4M3 encoder is compared with a brute-force nearest-value
search over the whole code table, ties to the even code, and saturation.
"""
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _same(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    both_nan = np.isnan(a) & np.isnan(b)
    eq = (a == b) & (np.signbit(a) == np.signbit(b))
    return bool(np.all(both_nan | eq))


def test_f16_decode_all_codes():
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    assert _same(oracle.decode(oracle.F16, codes), ref)


def test_bf16_decode_all_codes():
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    t = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16)
    ref = t.to(torch.float64).numpy()
    assert _same(oracle.decode(oracle.BF16, codes), ref)


def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    t = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn)
    ref = t.to(torch.float64).numpy()
    assert _same(oracle.decode(oracle.E4M3, codes), ref)


def test_e4m3_decode_format_points():
    # OCP 8-bit floating point, E4M3: bias 7, 3 mantissa bits, S.1111.111 = NaN
    points = {0x00: 0.0, 0x80: -0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9,
              0x08: 2.0 ** -6, 0x38: 1.0, 0x3c: 1.5, 0x7e: 448.0, 0xfe: -448.0,
              0x77: 240.0, 0x40: 2.0}
    for code, val in points.items():
        got = oracle.decode(oracle.E4M3, np.array([code], np.uint8))[0]
        assert got == val and math.copysign(1, got) == math.copysign(1, val), hex(code)
    assert np.isnan(oracle.decode(oracle.E4M3, np.array([0x7f, 0xff], np.uint8))).all()
    # 126 distinct positive finite values
    vals = oracle.decode(oracle.E4M3, np.arange(0x01, 0x7f, dtype=np.uint8))
    assert len(np.unique(vals)) == 126 and np.all(np.diff(vals) > 0)


def _brute_encode(y):
    """Nearest finite E4M3 value by search; ties go to the even code."""
    codes = np.arange(0, 0x7f, dtype=np.uint8)            # non-negative finite
    vals = oracle.decode(oracle.E4M3, codes)
    out = np.empty(len(y), np.uint8)
    for i, x in enumerate(np.asarray(y, np.float64)):
        sign = 0x80 if math.copysign(1.0, x) < 0 else 0
        a = abs(x)
        if a >= 448.0:
            out[i] = sign | 0x7e
            continue
        d = np.abs(vals - a)
        best = np.flatnonzero(d == d.min())
        if len(best) > 1:
            best = [c for c in best if c % 2 == 0]
        out[i] = sign | int(codes[best[0]])
    return out


def test_e4m3_encode_matches_brute_force():
    rng = np.random.default_rng(11)
    vals = oracle.decode(oracle.E4M3, np.arange(0, 0x7f, dtype=np.uint8))
    mids = (vals[1:] + vals[:-1]) / 2                       # exact ties
    y = np.concatenate([
        rng.standard_normal(20000) * 40,
        rng.standard_normal(5000) * 2.0 ** -7,
        mids, -mids,
        np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
        np.nextafter(mids.astype(np.float32), np.float32(0)),
        vals, -vals, [0.0, -0.0, 447.9, 448.0, 460.0, 479.9, 480.0, 1e30],
    ]).astype(np.float32)
    assert np.array_equal(oracle.encode_e4m3(y), _brute_encode(y))


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(12)
    y = np.concatenate([rng.standard_normal(50000) * 30,
                        rng.uniform(-464, 464, 20000),
                        rng.standard_normal(20000) * 2.0 ** -8]).astype(np.float32)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.encode_e4m3(y), ref)


def test_e4m3_encode_saturates_and_keeps_sign():
    y = np.array([448.0, 449.0, 480.0, 1e9, np.inf, -1e9, -np.inf, 0.0, -0.0,
                  2.0 ** -10, -(2.0 ** -10), 3 * 2.0 ** -11, 1.5 * 2.0 ** -9,
                  2.5 * 2.0 ** -9], np.float32)
    got = oracle.encode_e4m3(y)
    # 2^-10 is half the smallest subnormal: the tie goes to the even code 0;
    # 1.5 and 2.5 units of 2^-9 are ties that go to 2 units
    assert list(got) == [0x7e, 0x7e, 0x7e, 0x7e, 0x7e, 0xfe, 0xfe, 0x00, 0x80,
                         0x00, 0x80, 0x01, 0x02, 0x02]


def test_e4m3_round_trip_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7f) != 0x7f], np.uint8)
    vals = oracle.decode(oracle.E4M3, codes).astype(np.float32)
    assert np.array_equal(oracle.encode_e4m3(vals), codes)
