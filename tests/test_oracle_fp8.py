"""Pins of the FP8 block-scaled weight oracle (oracle/fp8.py) against things
other than itself: torch's float8_e4m3fn conversion, the E4M3 format's
landmark values, the block structure of the scale grid, and a library-built
expansion of the dequantised GEMM."""
import numpy as np
import pytest
import torch

from oracle import fp8 as of


def test_decoder_matches_torch_on_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = of.decode(codes.numpy())
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2  # S.1111.111 only: E4M3 has no infinities
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


@pytest.mark.parametrize("code,value", [
    (0x7E, 448.0),          # largest finite value
    (0x08, 2.0 ** -6),      # smallest normal
    (0x07, 7 * 2.0 ** -9),  # largest subnormal
    (0x01, 2.0 ** -9),      # smallest subnormal
    (0x38, 1.0),
    (0xB8, -1.0),
    (0x3C, 1.5),
    (0x00, 0.0),
])
def test_format_landmarks(code, value):
    assert of.e4m3_value(code) == value


def test_negative_zero_and_nan():
    assert of.e4m3_value(0x80) == 0.0 and np.signbit(of.e4m3_value(0x80))
    assert np.isnan(of.e4m3_value(0x7F)) and np.isnan(of.e4m3_value(0xFF))
    assert not np.isnan(of.e4m3_value(0x7E)) and not np.isnan(of.e4m3_value(0x77))


def _codes(rng, shape):
    q = rng.integers(0, 256, size=shape).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x3A  # no NaN codes in weights
    return q


def test_unit_scales_give_the_decoder():
    rng = np.random.default_rng(0)
    q = _codes(rng, (130, 200))
    W = of.dequantize(q, np.ones((2, 2)))
    assert np.array_equal(W, of.decode(q))


@pytest.mark.parametrize("bi,bj", [(0, 0), (1, 0), (0, 1), (1, 2)])
def test_one_scaled_block(bi, bj):
    """A scale grid of ones except 2^5 at block (bi, bj): exactly the elements
    of rows [128 bi, 128 bi + 128) x columns [128 bj, 128 bj + 128) (cut at the
    ragged edges of a 200 x 300 matrix) are multiplied by 32 -- a transposed
    grid index or another block size fails."""
    rng = np.random.default_rng(1)
    q = _codes(rng, (200, 300))
    s = np.ones((2, 3))
    s[bi, bj] = 32.0
    ratio = of.dequantize(q, s)
    base = of.decode(q)
    mask = np.zeros(q.shape, dtype=bool)
    mask[128 * bi:128 * bi + 128, 128 * bj:128 * bj + 128] = True
    nz = base != 0
    assert np.array_equal(ratio[mask & nz] / base[mask & nz], np.full((mask & nz).sum(), 32.0))
    assert np.array_equal(ratio[~mask], base[~mask])


def test_scale_grid_shape_is_checked():
    q = np.zeros((129, 256), dtype=np.uint8)
    with pytest.raises(ValueError):
        of.dequantize(q, np.ones((1, 2)))


def test_gemm_against_library_expansion():
    """x @ W^T with W built by torch's float8 decoding and a Kronecker
    expansion of the scale grid (numpy), not by the oracle's own code."""
    rng = np.random.default_rng(2)
    R, N, K = 5, 260, 400
    q = _codes(rng, (N, K))
    s = rng.uniform(0.001, 0.01, size=(3, 4)).astype(np.float32).astype(np.float64)
    x = rng.standard_normal((R, K))
    dec = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    grid = np.kron(s, np.ones((128, 128)))[:N, :K]
    ref = x @ (dec * grid).T
    got = of.gemm(x, q, s)
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-13)


def test_dequantised_product_is_exact():
    """An e4m3 value (4 significant bits) times an fp32 scale (24 bits) is
    exact in float64: the product times the inverse power-of-two part of the
    scale recovers the code's value."""
    q = np.arange(256, dtype=np.uint8).reshape(16, 16)
    q[(q & 0x7F) == 0x7F] = 0
    s = np.array([[np.float32(0.0123456789)]], dtype=np.float64)
    W = of.dequantize(q, s)
    assert np.array_equal(W / s[0, 0], of.decode(q))
