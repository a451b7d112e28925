"""MXFP8 (E4M3 elements, E8M0 scale per 32 elements) on the CPU, in float64.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this module;
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
use it.

The pages ask for "group-aware MXFP8 quantisation" of expert activations and an
"MXFP8 grouped GEMM" for the expert matmuls (Blog [1], section "What dropless
MoE needs" and section "Optimisation 1: grouped GEMM"), and list MXFP8 as the
Blackwell low-precision recipe (Reading [3], contribution 3).  They never give
the encoding, so this module follows the published MX definition: OCP
Microscaling Formats (MX) Specification v1.0 -- the FP8 E4M3 element format
(bias 7, subnormals, no infinities, S.1111.111 is NaN, largest normal 448), the
E8M0 scale (an unbiased power-of-two exponent stored with bias 127, 0xFF is
NaN), and its FP32 -> MX conversion: shared exponent
``X = floor(log2(max_i |V_i|)) - emax_elem`` with ``emax_elem = 8`` for E4M3,
element codes ``P_i = RNE(V_i / 2^X)`` clamped to the largest normal.

Readings taken where the definition is silent (each also listed with the design's other readings):
* an all-zero block (amax == 0) gets scale byte 127 (2^0) and zero codes;
* X is clamped to the E8M0 range [-127, 127];
* the sign of a zero is kept (-0 encodes as 0x80);
* "group-aware": a 32-element block never holds elements of two experts.  For
  the row-wise scales of the forward path (blocks run along K inside one row,
  and a row belongs to exactly one expert) that holds by construction.

[1] "Accelerating Dropless MoE Training in JAX with NVIDIA Transformer Engine"
    (zhiding.cn rewrite of the NVIDIA technical blog).
[3] Deep reading of arXiv 2603.07685 (paper-daily.com), MoE training systems.

parity pinned: tests/test_oracle_mxfp8.py (format table from the definition,
torch.float8_e4m3fn casts of in-range values, idempotence, closed-form scales,
golden points in tests/golden/e4m3_points.txt; the column-wise round trip against
the row-wise one of the transpose, and group separation under the E4M3 bound).
"""

from __future__ import annotations

import numpy as np

BLOCK = 32          # elements per E8M0 scale
E4M3_EMAX = 8       # exponent of the largest E4M3 normal (448 = 1.75 * 2^8)
E4M3_MAX = 448.0
E8M0_BIAS = 127


def e4m3_decode(code: int) -> float:
    """Value of one E4M3 byte, straight from the bit-field definition."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:
        return sign * (man / 8.0) * 2.0 ** (1 - 7)        # subnormal: 0.mmm * 2^-6
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


# Non-negative finite values, indexed by code 0x00..0x7E; strictly increasing.
E4M3_POS = np.array([e4m3_decode(c) for c in range(0x7F)], dtype=np.float64)
E4M3_ALL = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(y: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even to E4M3 with saturation to +-448.  float64 in, uint8 codes out.

    The nearest representable magnitude is found by bracketing |y| between two
    neighbouring table entries; an exact tie picks the entry whose code has an
    even last mantissa bit.  Magnitudes at or above 448 saturate to 448.
    """
    y = np.asarray(y, dtype=np.float64)
    if np.isnan(y).any():
        raise ValueError("NaN input is outside the quantiser's domain")
    mag = np.abs(y)
    sign = np.signbit(y)
    hi = np.searchsorted(E4M3_POS, mag, side="left")           # E4M3_POS[hi] >= mag
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - E4M3_POS[lo]
    d_hi = E4M3_POS[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(mag >= E4M3_MAX, 0x7E, code)
    return (code | np.where(sign, 0x80, 0)).astype(np.uint8)


def shared_exponent(amax: np.ndarray) -> np.ndarray:
    """X = floor(log2(amax)) - 8, clamped to [-127, 127]; amax == 0 gives X = 0.

    floor(log2) is read off an exact frexp decomposition (amax = m * 2^e with
    m in [0.5, 1) gives floor(log2 amax) = e - 1), so no logarithm is rounded.
    """
    amax = np.asarray(amax, dtype=np.float64)
    _, e = np.frexp(amax)
    x = (e.astype(np.int64) - 1) - E4M3_EMAX
    x = np.clip(x, -127, 127)
    return np.where(amax == 0.0, 0, x)


def quantize_rowwise(a: np.ndarray):
    """Row-wise MXFP8 of a [rows, K] matrix (K % 32 == 0) -> (codes u8 [rows,K], scales u8 [rows,K/32])."""
    a = np.asarray(a, dtype=np.float64)
    rows, K = a.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 32")
    blocks = a.reshape(rows, K // BLOCK, BLOCK)
    amax = np.abs(blocks).max(axis=-1)
    X = shared_exponent(amax)
    scaled = blocks * np.exp2(-X.astype(np.float64))[..., None]   # exact: power-of-two scaling
    codes = e4m3_encode(scaled).reshape(rows, K)
    scales = (X + E8M0_BIAS).astype(np.uint8)
    return codes, scales


def dequantize_rowwise(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Exact float64 values code * 2^(scale - 127)."""
    rows, K = codes.shape
    vals = E4M3_ALL[codes.astype(np.int64)].reshape(rows, K // BLOCK, BLOCK)
    mult = np.exp2(scales.astype(np.float64) - E8M0_BIAS)[..., None]
    return (vals * mult).reshape(rows, K)


def quantize_colwise_grouped(a: np.ndarray, offsets: np.ndarray):
    """Column-wise, group-aware MXFP8 of a [rows, K] matrix whose rows are split into
    contiguous expert groups by ``offsets`` [E+1].

    Blocks run down a column over 32 consecutive rows and restart at every group
    start; a group's last partial block is padded with zeros (which never change
    its amax).  Returns codes u8 [rows, K] and scales u8 [n_blocks, K] where the
    blocks of group e start at block row sum_{e'<e} ceil(count_e'/32).
    """
    a = np.asarray(a, dtype=np.float64)
    rows, K = a.shape
    offsets = np.asarray(offsets, dtype=np.int64)
    E = len(offsets) - 1
    nb = [(int(offsets[e + 1] - offsets[e]) + BLOCK - 1) // BLOCK for e in range(E)]
    codes = np.zeros((rows, K), dtype=np.uint8)
    scales = np.zeros((sum(nb), K), dtype=np.uint8)
    brow = 0
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        for b in range(nb[e]):
            r0, r1 = lo + b * BLOCK, min(lo + (b + 1) * BLOCK, hi)
            blk = a[r0:r1, :]
            X = shared_exponent(np.abs(blk).max(axis=0))
            codes[r0:r1, :] = e4m3_encode(blk * np.exp2(-X.astype(np.float64))[None, :])
            scales[brow, :] = (X + E8M0_BIAS).astype(np.uint8)
            brow += 1
    return codes, scales


def dequantize_colwise_grouped(codes: np.ndarray, scales: np.ndarray, offsets: np.ndarray) -> np.ndarray:
    """Exact float64 values of a column-wise group-aware quantisation: row r of
    group e, column c decodes as code * 2^(scale[block row of r, c] - 127), the
    block rows numbered as in ``quantize_colwise_grouped``."""
    codes = np.asarray(codes)
    rows, K = codes.shape
    offsets = np.asarray(offsets, dtype=np.int64)
    out = np.zeros((rows, K), dtype=np.float64)
    brow = 0
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        for r0 in range(lo, hi, BLOCK):
            r1 = min(r0 + BLOCK, hi)
            mult = np.exp2(scales[brow].astype(np.float64) - E8M0_BIAS)
            out[r0:r1] = E4M3_ALL[codes[r0:r1].astype(np.int64)] * mult[None, :]
            brow += 1
    return out
