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

The activations of such a GEMM enter the tensor cores as e4m3 too (the
runtime's compute representation; reading): each 128-wide k-tile of a token's
bf16 activation row is scaled by the power of two 2^E with the smallest E such
that max|x| <= 448 * 2^E, and represented as 2^E (hi + lo) with
hi = RNE_e4m3(x / 2^E) and lo = RNE_e4m3(x / 2^E - hi) (round to nearest,
ties to even, saturating).  Because a bf16 value has 8 significant bits and an
e4m3 value 4, the two terms reproduce every element of magnitude >= 2^(E-2)
exactly; smaller ones are off by at most 2^(E-10) (the e4m3 subnormal step is
2^-9).  ``split_activations`` states this; ``gemm_split`` is the GEMM on the
represented activations.

Pins (tests/test_oracle_fp8.py): the decoder against torch's float8_e4m3fn
conversion on all 256 codes and at the format's landmarks (448, 2^-6, 2^-9,
±0, NaN); dequantisation with unit scales is the decoder; a scale grid that is
one except for a single block multiplies exactly that block's elements
(ragged edges included); the GEMM against x @ (decoded q * Kronecker-expanded
scale grid)^T built from library routines; the rounding function against
torch's float8 conversion on random and tie values; the split's exponent
minimality, exactness region and error bound.
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


# ---------------------------------------------------------------------------
# activations as two e4m3 terms per 128-wide k-tile
# ---------------------------------------------------------------------------
_POS = np.array(sorted(v for v in _TABLE[:0x7F] if v >= 0.0))  # the 127 finite non-negative values, codes 0..126


def e4m3_round(v) -> np.ndarray:
    """Nearest E4M3 value to each float (ties to the even code, i.e. the
    value whose mantissa's last bit is 0), saturating at +-448."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), 448.0)
    hi = np.searchsorted(_POS, a, side="left")          # first value >= a
    hi = np.minimum(hi, len(_POS) - 1)
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = a - _POS[lo], _POS[hi] - a
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    return np.copysign(_POS[pick], v)


def split_exponent(amax: float) -> int:
    """Smallest integer E with amax <= 448 * 2^E (0 for amax = 0)."""
    if amax == 0.0:
        return 0
    E = int(np.floor(np.log2(amax / 448.0)))
    while amax > 448.0 * 2.0 ** E:
        E += 1
    while amax <= 448.0 * 2.0 ** (E - 1):
        E -= 1
    return E


def split_activations(x):
    """x [R, K] (bf16 values) -> (E [R, ceil(K/128)] int, hi, lo [R, K] float64
    e4m3 values) with x ~= 2^E (hi + lo) per 128-wide k-tile."""
    x = np.asarray(x, dtype=np.float64)
    R, K = x.shape
    nkb = -(-K // BLOCK)
    E = np.zeros((R, nkb), dtype=np.int64)
    hi = np.zeros_like(x)
    lo = np.zeros_like(x)
    for r in range(R):
        for kb in range(nkb):
            sl = slice(kb * BLOCK, min(K, (kb + 1) * BLOCK))
            e = split_exponent(float(np.abs(x[r, sl]).max()))
            v = x[r, sl] / 2.0 ** e
            h = e4m3_round(v)
            E[r, kb] = e
            hi[r, sl] = h
            lo[r, sl] = e4m3_round(v - h)
    return E, hi, lo


def represented_activations(x) -> np.ndarray:
    """2^E (hi + lo): the activations the FP8 GEMM multiplies."""
    E, hi, lo = split_activations(x)
    scale = np.repeat(2.0 ** E.astype(np.float64), BLOCK, axis=1)[:, :np.asarray(x).shape[1]]
    return scale * (hi + lo)


def gemm_split(x, q, scale) -> np.ndarray:
    """x [R, K] @ W^T with x in its two-term e4m3 form and W dequantised."""
    return represented_activations(x) @ dequantize(q, scale).T
