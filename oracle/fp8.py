"""FP8 block-scaled weights -- oracle, test infrastructure only.

"M7.6 - DeepSeek MTP: Sequential Modules, Teacher Forcing, and Speculative
Runtime" §0x03C (the layered numerical contract): the released weights are
stored as FP8 with block-scale metadata, while the compute representation is
the runtime's choice.  Reading: the FP8 format is OCP FP8 E4M3 (sign, four
exponent bits with bias 7, three mantissa bits, subnormals, no infinities,
S.1111.111 = NaN) and the scale metadata one fp32 factor per 128 x 128 block
of the [out, in] matrix, so the represented weight is

    W[m, k] = e4m3(q[m, k]) * scale[m // 128, k // 128]

taken exactly (an e4m3 value has 4 significant bits and the scale 24, so the
float64 product is exact).  The FP8 draft step is the draft-step oracle run on
these exact weights.

Pins (tests/test_oracle_fp8.py): the decoder against torch's float8_e4m3fn
conversion on all 256 codes and at the format's landmarks (448, 2^-6, 2^-9,
±0, NaN); dequantisation with unit scales is the decoder; a scale grid that is
one except for a single block multiplies exactly that block's elements
(ragged edges included); the GEMM against x @ (decoded q * Kronecker-expanded
scale grid)^T built from library routines.
"""
from __future__ import annotations

import numpy as np

BLOCK = 128
LINEAR_MAPS = ("eh_proj", "wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


def e4m3_value(code: int) -> float:
    """Value of one E4M3 code (0..255) from the format's definition."""
    code = int(code)
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** (1 - 7)  # subnormal
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def decode(q) -> np.ndarray:
    """E4M3 codes (uint8 array) -> float64 values."""
    return _TABLE[np.asarray(q, dtype=np.uint8)]


def dequantize(q, scale) -> np.ndarray:
    """W = e4m3(q) * scale[m // 128, k // 128], float64 (exact)."""
    q = np.asarray(q, dtype=np.uint8)
    scale = np.asarray(scale, dtype=np.float64)
    n, k = q.shape
    rows = np.arange(n) // BLOCK
    cols = np.arange(k) // BLOCK
    if scale.shape != (rows[-1] + 1, cols[-1] + 1):
        raise ValueError(f"scale grid {scale.shape} does not match [{n}, {k}] in {BLOCK}x{BLOCK} blocks")
    return decode(q) * scale[rows][:, cols]


def gemm(x, q, scale) -> np.ndarray:
    """x [R, K] @ W^T with W the dequantised [N, K] matrix (float64)."""
    return np.asarray(x, dtype=np.float64) @ dequantize(q, scale).T


def draft_weights(W: dict, fp8: dict) -> dict:
    """The draft-step oracle's weight dict with the module's linear maps
    replaced by their exact dequantised FP8 forms; fp8[name] = (q, scale)."""
    out = dict(W)
    for name in LINEAR_MAPS:
        q, s = fp8[name]
        out[name] = [dequantize(np.asarray(q), np.asarray(s))]
    return out
