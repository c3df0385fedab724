"""Pins of the oracle's MXFP8 quantiser: the E4M3 code table, round-to-nearest-
even against torch's float8_e4m3fn cast (a library routine), the format's
printed encoding points (tests/golden/e4m3_points.txt) and the block-scale
rule with its error bounds."""
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_points.txt")


def test_decode_encode_roundtrip_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    vals = O.e4m3_decode(codes)
    finite = ~np.isnan(vals)
    assert finite.sum() == 254                      # 0x7F and 0xFF are NaN
    back = O.e4m3_encode(vals[finite])
    np.testing.assert_array_equal(back, codes[finite])
    assert np.nanmax(vals) == 448.0 and np.nanmin(vals) == -448.0


def test_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    tv = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ov = O.e4m3_decode(codes.numpy())
    np.testing.assert_array_equal(np.isnan(tv), np.isnan(ov))
    m = ~np.isnan(ov)
    np.testing.assert_array_equal(tv[m], ov[m])


def test_encode_matches_torch_rne_in_range():
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.standard_normal(200000) * 50,
        rng.standard_normal(50000) * 0.01,          # subnormal range
        rng.uniform(-448, 448, 50000),
    ])
    v = np.clip(v, -448, 448)
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_encode(v)
    # torch keeps the sign of zero the same way
    np.testing.assert_array_equal(got, want)


def test_midpoints_round_to_even_and_saturate():
    vals = O.e4m3_decode(np.arange(0, 0x7E, dtype=np.uint8))   # positive finite, ascending
    mids = (vals[:-1] + vals[1:]) / 2
    got = O.e4m3_encode(mids)
    lo = np.arange(0, 0x7D)
    want = np.where(lo % 2 == 0, lo, lo + 1)        # even mantissa == even code
    np.testing.assert_array_equal(got, want.astype(np.uint8))
    assert O.e4m3_encode(np.array([448.0, 463.99, 464.0, 1e6, -1e6])).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]


def test_golden_points():
    """Encodings printed in the OCP 8-bit floating point specification v1.0
    (E4M3 column of its format table)."""
    n = 0
    with open(GOLDEN) as fh:
        for line in fh:
            line = line.split("#")[0].strip()
            if not line:
                continue
            val, code = line.split()
            v = float.fromhex(val) if val.startswith(("0x", "-0x")) else float(val)
            c = int(code, 16)
            assert O.e4m3_encode(np.array([v]))[0] == c, line
            assert O.e4m3_decode(np.array([c]))[0] == v, line
            n += 1
    assert n >= 8


def test_block_scale_rule_and_error_bound():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((64, 256)) * np.exp2(rng.integers(-20, 20, size=(64, 1)))
    v[3, 32:64] = 0.0                                  # an all-zero block
    codes, scales = O.mxfp8_quantize(v, axis=-1)
    assert scales.shape == (64, 8)
    assert scales[3, 1] == 0 and np.all(codes[3, 32:64] == 0)
    blocks = v.reshape(64, 8, 32)
    amax = np.abs(blocks).max(-1)
    nz = amax > 0
    e = scales.astype(np.int64) - 127
    # largest element lands in [256, 512) after scaling: 2^(e+8) <= amax < 2^(e+9)
    assert np.all(np.exp2(e[nz] + 8.0) <= amax[nz]) and np.all(amax[nz] < np.exp2(e[nz] + 9.0))
    deq = O.mxfp8_dequantize(codes, scales, axis=-1)
    X = np.repeat(np.exp2(e.astype(np.float64)), 32, axis=-1)
    r = np.abs(v) / X
    err = np.abs(deq - v)
    normal = (r >= 2.0 ** -6) & (r <= 448.0)
    sub = r < 2.0 ** -6
    sat = r > 448.0
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(v[normal]))
    assert np.all(err[sub] <= 2.0 ** -10 * X[sub])
    assert np.all(np.abs(deq[sat]) == 448.0 * X[sat])


def test_quantize_other_axis_is_transpose():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((64, 96))
    c0, s0 = O.mxfp8_quantize(v, axis=0)
    c1, s1 = O.mxfp8_quantize(v.T, axis=-1)
    np.testing.assert_array_equal(c0, c1.T)
    np.testing.assert_array_equal(s0, s1.T)


def test_block_must_be_multiple_of_32():
    with pytest.raises(ValueError):
        O.mxfp8_quantize(np.zeros((2, 33)))
