"""NVFP4 (E2M1 elements, one E4M3 scale per 16 elements, one fp32 scale per tensor)
on the CPU.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this module;
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
use it.

Reading [3] ("Deep reading of arXiv 2603.07685", contribution 3) names NVFP4 as
the Blackwell low-precision recipe beside MXFP8 and [1] lists FP4 among its
planned work; neither defines it.  This module follows NVIDIA's published NVFP4
description: FP4 E2M1 elements (1 sign bit, 2 exponent bits with bias 1, 1
mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), a block of 16 consecutive
elements sharing one FP8 E4M3 scale, and a second, fp32 scale for the whole
tensor so that the block scales use the E4M3 range.

Readings taken where the description leaves the arithmetic open, written so that
every rounding that decides a code happens in fp32, in this order, on both sides:
* tensor encode scale g = 2688 / amax(tensor) (2688 = 448 * 6, the largest E4M3
  times the largest E2M1), one fp32 division; an all-zero tensor gets g = 1;
* block scale: s = E4M3(fp32(fp32(amax_block / 6) * g)), round to nearest even,
  saturating at 448 (an unsigned E4M3: the sign bit is never set);
* element: y = fp32(v * fp32(g / s_value)) (y = v * 0 when s decodes to 0), then
  E2M1 round to nearest even (ties to the even code), saturating at 6, the sign
  of zero kept;
* decoded value = e2m1 * s_value / g (exact);
* storage: codes packed two per byte, element 2i in the low nibble; scales
  [rows, K/16] bytes; the tensor scale g as one fp32.

parity pinned: tests/test_oracle_nvfp4.py (E2M1 table from the bit fields, hand-
worked blocks in tests/golden/nvfp4_blocks.txt, RNE midpoints, error bound,
power-of-two invariance of the two-level scale, packing order).
"""

from __future__ import annotations

import numpy as np

from oracle import mxfp8

BLOCK = 16
E2M1_MAX = 6.0
TENSOR_NUM = np.float32(448.0 * 6.0)


def e2m1_decode(code: int) -> float:
    """Value of one 4-bit E2M1 code from its bit fields."""
    code = int(code) & 0xF
    sign = -1.0 if code & 0x8 else 1.0
    exp = (code >> 1) & 0x3
    man = code & 0x1
    if exp == 0:
        return sign * (man / 2.0)                       # subnormal: 0.m * 2^(1 - 1)
    return sign * (1.0 + man / 2.0) * 2.0 ** (exp - 1)


E2M1_POS = np.array([e2m1_decode(c) for c in range(8)], dtype=np.float64)    # 0 .. 6
E2M1_ALL = np.array([e2m1_decode(c) for c in range(16)], dtype=np.float64)


def e2m1_encode(y: np.ndarray) -> np.ndarray:
    """Round to nearest even E2M1 with saturation to +-6; float in, 4-bit codes out.
    An exact tie picks the code with an even last (mantissa) bit."""
    y = np.asarray(y, dtype=np.float64)
    mag = np.abs(y)
    hi = np.minimum(np.searchsorted(E2M1_POS, mag, side="left"), 7)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - E2M1_POS[lo]
    d_hi = E2M1_POS[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(mag >= E2M1_MAX, 7, code)
    return (code | np.where(np.signbit(y), 0x8, 0)).astype(np.uint8)


def tensor_scale(a: np.ndarray) -> np.float32:
    """g = 2688 / amax(tensor) in fp32 (1 for an all-zero tensor)."""
    amax = np.float32(np.abs(np.asarray(a, dtype=np.float32)).max()) if np.size(a) else np.float32(0)
    return np.float32(1.0) if amax == 0 else np.float32(TENSOR_NUM / amax)


def quantize(a: np.ndarray, g: np.float32 | None = None):
    """NVFP4 of a [rows, K] matrix (K % 16 == 0) in the recipe above.

    Returns (codes u8 [rows, K/2] packed, scales u8 [rows, K/16] E4M3, g fp32)."""
    a = np.asarray(a, dtype=np.float32)
    rows, K = a.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 16")
    if g is None:
        g = tensor_scale(a)
    g = np.float32(g)
    blocks = a.reshape(rows, K // BLOCK, BLOCK)
    amax = np.abs(blocks).max(axis=-1).astype(np.float32)
    sf = (amax / np.float32(6.0)).astype(np.float32)
    sf = (sf * g).astype(np.float32)
    s_code = mxfp8.e4m3_encode(sf.astype(np.float64))                 # sf >= 0: sign bit clear
    s_val = mxfp8.E4M3_ALL[s_code.astype(np.int64)].astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(s_val == 0, np.float32(0), (g / s_val).astype(np.float32)).astype(np.float32)
    y = (blocks * inv[..., None]).astype(np.float32)
    c = e2m1_encode(y.astype(np.float64)).reshape(rows, K)
    packed = (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    return packed, s_code, g


def unpack(codes: np.ndarray) -> np.ndarray:
    """[rows, K/2] packed bytes -> [rows, K] 4-bit codes (element 2i from the low nibble)."""
    codes = np.asarray(codes, dtype=np.uint8)
    out = np.empty((codes.shape[0], codes.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = codes & 0xF
    out[:, 1::2] = codes >> 4
    return out


def dequantize(codes: np.ndarray, scales: np.ndarray, g) -> np.ndarray:
    """Exact float64 values e2m1 * s / g."""
    c = unpack(codes)
    rows, K = c.shape
    vals = E2M1_ALL[c.astype(np.int64)].reshape(rows, K // BLOCK, BLOCK)
    s = mxfp8.E4M3_ALL[np.asarray(scales).astype(np.int64)][..., None]
    return (vals * s / np.float64(g)).reshape(rows, K)
