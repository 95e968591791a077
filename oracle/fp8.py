"""FP8 E4M3 block quantization for the oracle (plain numpy, written from the format's
definition).

TEST INFRASTRUCTURE ONLY, like the rest of this package: the tests and the benchmark's
CPU-baseline leg use it; the CUDA library never does.

The method ("FlashAttention-3: Warp Specialization and the 75% FLOPS Barrier on Hopper",
"FP8 Block Quantization"): each 128-row tile of Q and of K gets its own fp32 scale, the tile's
largest magnitude divided by 448 (the largest finite E4M3 value), and its elements are divided
by that scale and rounded to E4M3. The score of a query in tile a against a key in tile b is
then scale_a * scale_b * (q8 . k8). The page's prose calls the scales per tile; that is the
reading taken here (one scale per 128-row block of one head, over all of its columns).

E4M3 (the "fn" variant): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no
infinities; exponent field 0 holds subnormals m * 2^-9, the all-ones pattern S.1111.111 is NaN,
and the largest finite magnitude is 1.75 * 2^8 = 448.
"""
from __future__ import annotations

import numpy as np

BLOCK_ROWS = 128
E4M3_MAX = 448.0


def e4m3_values() -> np.ndarray:
    """Value of each of the 256 codes as float64 (NaN for the two NaN codes)."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = sign * m * 2.0 ** -9
        else:
            vals[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_VALUES = e4m3_values()
# Non-negative finite codes 0x00 .. 0x7E in increasing order of value.
_POS = _VALUES[:0x7F]


def e4m3_round(x) -> np.ndarray:
    """Round float32 values to E4M3 codes (uint8): nearest value, ties to the even code
    (mantissa LSB 0), magnitudes beyond 448 saturate to 448, sign kept (-0 for negative
    values that round to zero). NaN inputs are not expected and are rejected."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    if np.isnan(x).any():
        raise ValueError("NaN input")
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.searchsorted(_POS, a, side="left")  # first code with value >= a
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _POS[lo]
    d_hi = _POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((hi & 1) == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)


def quantize_blocks(x_bf16_bits: np.ndarray, block: int = BLOCK_ROWS):
    """Block-quantize x [planes, N, d] (bf16 bit patterns) to E4M3.

    For each plane and each block of `block` rows (the last one may be shorter):
      amax  = max |x| over the block (fp32, exact),
      scale = amax / 448 in fp32 (0 for an all-zero block),
      code  = e4m3_round(x / scale) with the division in fp32 (code 0 when scale is 0).
    Returns (codes uint8 [planes, N, d], scales float32 [planes, ceil(N/block)]).
    """
    bits = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
    x = (bits.astype(np.uint32) << 16).view(np.float32)
    planes, N, d = x.shape
    nb = (N + block - 1) // block
    codes = np.zeros((planes, N, d), dtype=np.uint8)
    scales = np.zeros((planes, nb), dtype=np.float32)
    for t in range(nb):
        blk = x[:, t * block:(t + 1) * block, :]
        amax = np.abs(blk).reshape(planes, -1).max(axis=1) if blk.shape[1] else \
            np.zeros(planes, np.float32)
        s = (amax.astype(np.float32) / np.float32(E4M3_MAX)).astype(np.float32)
        scales[:, t] = s
        for pl in range(planes):
            if s[pl] == 0:
                continue
            y = (blk[pl] / s[pl]).astype(np.float32)
            codes[pl, t * block:(t + 1) * block, :] = e4m3_round(y)
    return codes, scales


def dequantize(codes: np.ndarray, scales: np.ndarray, block: int = BLOCK_ROWS) -> np.ndarray:
    """codes [planes, N, d] and scales [planes, nblocks] -> float64 values code_value * scale
    (exact in float64: a 4-significant-bit value times a 24-bit scale)."""
    codes = np.asarray(codes, dtype=np.uint8)
    planes, N, d = codes.shape
    rows_scale = np.repeat(np.asarray(scales, dtype=np.float64), block, axis=1)[:, :N]
    return _VALUES[codes] * rows_scale[:, :, None]
