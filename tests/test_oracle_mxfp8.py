"""Pins for the oracle's MXFP8 quantiser (CPU only).

Pinned against: hand-worked E4M3 code points from the format definition
(tests/golden/e4m3_points.txt), PyTorch's own float32 -> float8_e4m3fn cast
(round-to-nearest-even) on in-range values and exact midpoints, closed-form
shared exponents, idempotence, and the per-element error bound of a 3-bit
mantissa.
"""

import math
import os

import numpy as np
import pytest
import torch

from oracle import mxfp8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _points():
    out = []
    for line in open(os.path.join(GOLDEN, "e4m3_points.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            c, v = line.split()
            out.append((int(c, 16), float(v)))
    return out


@pytest.mark.parametrize("code,value", _points())
def test_e4m3_golden_points(code, value):
    got = mxfp8.e4m3_decode(code)
    if math.isnan(value):
        assert math.isnan(got)
    else:
        assert got == value and math.copysign(1, got) == math.copysign(1, value)
        assert mxfp8.e4m3_encode(np.array([value]))[0] == code


def test_e4m3_table_shape():
    vals = mxfp8.E4M3_POS
    assert len(vals) == 127 and vals[0] == 0 and vals[-1] == 448.0
    assert (np.diff(vals) > 0).all()
    assert np.isnan(mxfp8.E4M3_ALL[0x7F]) and np.isnan(mxfp8.E4M3_ALL[0xFF])
    assert np.isfinite(mxfp8.E4M3_ALL).sum() == 254


def test_e4m3_matches_torch_cast_in_range():
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.standard_normal(20000) * 50,
        rng.uniform(-448, 448, 5000),
        rng.standard_normal(5000) * 1e-3,                  # subnormal range
    ]).astype(np.float32)
    # exact midpoints between neighbouring codes: the tie-to-even rule decides them
    mids = ((mxfp8.E4M3_POS[:-1] + mxfp8.E4M3_POS[1:]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids, np.float32([0.0, -0.0])])
    v = np.clip(v, -448, 448)
    ours = mxfp8.e4m3_encode(v.astype(np.float64))
    theirs = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (ours == theirs).all()


def test_e4m3_saturates():
    v = np.array([448.0, 449.0, 463.9, 464.0, 500.0, 1e6, -1e6])
    assert mxfp8.e4m3_encode(v).tolist() == [0x7E] * 5 + [0x7E, 0xFE]


def test_e4m3_roundtrip_all_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert (mxfp8.e4m3_encode(mxfp8.E4M3_ALL[codes]) == codes).all()


@pytest.mark.parametrize("amax,byte", [(1.0, 119), (448.0, 127), (0.75, 118), (3.0, 120),
                                       (511.9, 127), (512.0, 128), (2.0 ** -130, 0),
                                       (0.0, 127), (2.0 ** 127, 246), (2.0 ** 140, 254)])
def test_shared_exponent_closed_form(amax, byte):
    assert int(mxfp8.shared_exponent(np.array([amax]))[0]) + 127 == byte


def test_quantize_rowwise_properties():
    rng = np.random.default_rng(5)
    a = rng.standard_normal((64, 256)) * np.exp(rng.uniform(-8, 8, (64, 1)))
    a[3, 32:64] = 0.0                                   # an all-zero block
    codes, scales = mxfp8.quantize_rowwise(a)
    assert codes.shape == a.shape and scales.shape == (64, 8)
    assert scales[3, 1] == 127 and (codes[3, 32:64] == 0).all()
    deq = mxfp8.dequantize_rowwise(codes, scales)
    # idempotence: quantising dequantised values reproduces the bytes
    c2, s2 = mxfp8.quantize_rowwise(deq)
    assert (c2 == codes).all() and (s2 == scales).all()
    # every non-zero block's largest element lands in [256, 448] before scaling back
    X = scales.astype(np.int64) - 127
    blocks = np.abs(a).reshape(64, 8, 32)
    top = blocks.max(-1) / np.exp2(X)
    nz = blocks.max(-1) > 0
    assert ((top[nz] >= 256) & (top[nz] < 512)).all()
    # error bound: half an ulp of a 3-bit mantissa (2^-4 relative) in the normal
    # range, 2^(X-10) absolute in the subnormal range, unless saturated
    err = np.abs(a - deq).reshape(64, 8, 32)
    bound = np.maximum(blocks * 2.0 ** -4, np.exp2(X - 10)[..., None])
    sat = blocks / np.exp2(X)[..., None] > 448
    assert (err[~sat] <= bound[~sat] * (1 + 1e-12)).all()
    assert (np.abs(deq).reshape(64, 8, 32)[sat] == 448 * np.exp2(X)[..., None].repeat(32, -1)[sat]).all()


def test_quantize_keeps_sign_of_zero():
    a = np.zeros((1, 32))
    a[0, 0] = -0.0
    a[0, 1] = 1.0
    codes, _ = mxfp8.quantize_rowwise(a)
    assert codes[0, 0] == 0x80 and codes[0, 2] == 0x00


def test_colwise_grouped_blocks_restart_per_group():
    rng = np.random.default_rng(9)
    offsets = np.array([0, 5, 5, 45, 46])                # groups of 5, 0, 40 and 1 rows
    a = rng.standard_normal((46, 64))
    codes, scales = mxfp8.quantize_colwise_grouped(a, offsets)
    assert scales.shape == (1 + 0 + 2 + 1, 64)
    # each block equals the row-wise quantisation of its zero-padded transpose
    blocks = [(0, 5), (5, 37), (37, 45), (45, 46)]
    for b, (r0, r1) in enumerate(blocks):
        pad = np.zeros((32, 64))
        pad[:r1 - r0] = a[r0:r1]
        c_t, s_t = mxfp8.quantize_rowwise(pad.T.copy())
        assert (scales[b] == s_t[:, 0]).all()
        assert (codes[r0:r1].T == c_t[:, :r1 - r0]).all()


def test_colwise_dequantize_matches_transposed_rowwise():
    """One group whose size is a multiple of 32: the column-wise round trip equals
    the row-wise round trip of the transpose (already pinned above)."""
    rng = np.random.default_rng(11)
    a = rng.standard_normal((96, 64)) * np.exp2(rng.integers(-6, 6, size=(96, 1)))
    codes, scales = mxfp8.quantize_colwise_grouped(a, np.array([0, 96]))
    got = mxfp8.dequantize_colwise_grouped(codes, scales, np.array([0, 96]))
    c_t, s_t = mxfp8.quantize_rowwise(a.T.copy())
    assert np.array_equal(got, mxfp8.dequantize_rowwise(c_t, s_t).T)


def test_colwise_dequantize_keeps_groups_apart():
    """Neighbouring groups of very different magnitude: each element comes back
    within the E4M3 half-ulp bound of its own group's block (a scale taken from
    the wrong group would flush the small group to zero or saturate it).  Values
    lie in [1, 1.5) times a power of two per group: normal range, no saturation."""
    rng = np.random.default_rng(12)
    offsets = np.array([0, 7, 7, 40, 41, 75])
    a = rng.uniform(1.0, 1.5, size=(75, 32)) * rng.choice([-1.0, 1.0], size=(75, 32))
    a[7:40] *= 2.0 ** 12
    a[41:75] *= 2.0 ** -12
    codes, scales = mxfp8.quantize_colwise_grouped(a, offsets)
    got = mxfp8.dequantize_colwise_grouped(codes, scales, offsets)
    assert (np.abs(got - a) <= np.abs(a) * 2.0 ** -4 + 1e-300).all()
    assert (got != 0).all()
