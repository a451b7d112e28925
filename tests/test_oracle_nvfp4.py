"""Pins for the NVFP4 oracle (CPU only): the E2M1 table from its bit fields,
hand-worked blocks (tests/golden/nvfp4_blocks.txt), round-to-nearest-even at
every midpoint, the error bound of the two-level scale, its invariance under a
power-of-two rescaling of the tensor, and the packing order."""

import os

import numpy as np

from oracle import mxfp8, nvfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_blocks.txt")


def test_e2m1_table_from_the_format():
    assert list(nvfp4.E2M1_POS) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert np.array_equal(nvfp4.E2M1_ALL[8:], -nvfp4.E2M1_POS)
    assert np.signbit(nvfp4.E2M1_ALL[8])                        # code 0x8 is -0


def test_golden_blocks():
    fields = {}
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            key, *vals = line.split()
            fields[key] = vals
    v = np.array([float(x) for x in fields["values"]], dtype=np.float32)[None, :]
    codes, scales, g = nvfp4.quantize(v)
    assert g == np.float32(fields["g"][0])
    assert [f"{b:02X}" for b in scales[0]] == fields["scales"]
    assert [f"{b:02X}" for b in codes[0]] == fields["codes"]


def test_e2m1_midpoints_round_to_even_and_saturate():
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    want = np.array([0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0])
    got = nvfp4.E2M1_ALL[nvfp4.e2m1_encode(mids).astype(np.int64)]
    assert np.array_equal(got, want)
    assert np.array_equal(nvfp4.E2M1_ALL[nvfp4.e2m1_encode(-mids).astype(np.int64)], -want)
    assert (nvfp4.e2m1_encode(np.array([6.0, 7.0, 1e30])) == 0x7).all()
    # just off a midpoint goes to the nearer value
    eps = 1e-6
    assert nvfp4.E2M1_ALL[nvfp4.e2m1_encode(np.array([0.25 + eps]))[0]] == 0.5
    assert nvfp4.E2M1_ALL[nvfp4.e2m1_encode(np.array([2.5 + eps]))[0]] == 3.0


def test_error_bound_of_the_two_level_scale():
    """Every element decodes within half an E2M1 step of its scaled value (the
    step at magnitude m is 0.5 below 2, 1 below 4, 2 up to 6) times s / g, plus the
    E4M3 rounding of the block scale when that pushes the block past 6."""
    rng = np.random.default_rng(3)
    a = (rng.standard_normal((64, 256)) * np.exp2(rng.integers(-8, 8, size=(64, 1)))).astype(np.float32)
    codes, scales, g = nvfp4.quantize(a)
    deq = nvfp4.dequantize(codes, scales, g)
    s = mxfp8.E4M3_ALL[scales.astype(np.int64)]
    y = np.abs(a.reshape(64, 16, 16).astype(np.float64)) * (np.float64(g) / s)[..., None]
    step = np.where(y < 2, 0.5, np.where(y < 4, 1.0, 2.0))
    over = np.maximum(y - 6.0, 0.0)                               # saturation: s rounded down
    bound = (step / 2 + over) * (s / np.float64(g))[..., None]
    err = np.abs(deq.reshape(64, 16, 16) - a.reshape(64, 16, 16))
    assert (err <= bound * (1 + 1e-6) + 1e-30).all()
    # a normal-range E4M3 scale is within 2^-4 of amax/6*g, so saturation stays below
    # 6 / (1 - 2^-4) = 6.4; subnormal scales (tiny blocks) are coarser
    normal = s >= 2.0 ** -6
    assert (over[normal] <= 0.4 + 1e-12).all()
    assert normal.mean() > 0.5


def test_power_of_two_rescaling_keeps_codes():
    rng = np.random.default_rng(4)
    a = rng.standard_normal((8, 64)).astype(np.float32)
    c0, s0, g0 = nvfp4.quantize(a)
    c1, s1, g1 = nvfp4.quantize(a * np.float32(2.0 ** 5))
    assert np.array_equal(c0, c1) and np.array_equal(s0, s1) and g1 == g0 / np.float32(32)
    assert np.array_equal(nvfp4.dequantize(c1, s1, g1), nvfp4.dequantize(c0, s0, g0) * 32)


def test_packing_order_and_zero_tensor():
    a = np.zeros((1, 16), dtype=np.float32)
    a[0, 0], a[0, 1] = 6.0, -1.0                                  # codes 0x7 and 0xA
    codes, _, _ = nvfp4.quantize(a)
    assert codes[0, 0] == 0xA7
    assert np.array_equal(nvfp4.unpack(codes)[0, :2], [0x7, 0xA])
    z, zs, zg = nvfp4.quantize(np.zeros((2, 32), dtype=np.float32))
    assert zg == 1 and (z == 0).all() and (zs == 0).all()
