"""Pins of the FP8 block-scaled weight oracle (oracle/fp8.py) against things
other than itself: torch's float8_e4m3fn conversion, the E4M3 format's
landmark values, the block structure of the scale grid, a library-built
expansion of the dequantised GEMM, and the two-term activation split's
exponent, exactness region and error bound."""
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


def test_rounding_matches_torch():
    """RNE to E4M3 against torch's float8_e4m3fn conversion on values spread
    over the whole range, and on every tie between neighbouring values."""
    rng = np.random.default_rng(3)
    v = rng.standard_normal(200000) * np.exp(rng.uniform(-14, 6.1, 200000))
    v = np.clip(v, -448.0, 448.0).astype(np.float32)
    vals = np.array(sorted(set(of.decode(np.arange(0, 127, dtype=np.uint8)).tolist())))
    ties = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    for t in (v, ties, -ties):
        ref = torch.from_numpy(t).to(torch.float8_e4m3fn).to(torch.float64).numpy()
        assert np.array_equal(of.e4m3_round(t.astype(np.float64)), ref)


def test_split_exponent_is_minimal():
    rng = np.random.default_rng(4)
    for amax in np.concatenate([rng.uniform(1e-6, 1e4, 500), [448.0, 224.0, 448.0 * 2 ** -7, 1.0, 2.0 ** -30]]):
        E = of.split_exponent(float(amax))
        assert amax <= 448.0 * 2.0 ** E and amax > 448.0 * 2.0 ** (E - 1)
    assert of.split_exponent(0.0) == 0


def _bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def test_split_is_exact_within_its_range_and_bounded_below():
    """x~ = x for every element of magnitude >= 2^(E-2); below that the
    error is at most 2^(E-10); hi and lo are e4m3 values."""
    rng = np.random.default_rng(5)
    x = _bf16(rng.standard_normal((6, 300)) * np.exp(rng.uniform(-12, 4, (6, 300))))
    E, hi, lo = of.split_activations(x)
    xt = of.represented_activations(x)
    s = np.repeat(2.0 ** E, 128, axis=1)[:, :300]
    big = np.abs(x) >= s / 4
    assert big.sum() > 100 and (~big).sum() > 100
    assert np.array_equal(xt[big], x[big])
    assert np.all(np.abs(xt - x) <= s * 2.0 ** -10)
    assert np.array_equal(of.e4m3_round(hi), hi) and np.array_equal(of.e4m3_round(lo), lo)


def test_split_of_e4m3_representable_values_has_no_low_term():
    """An activation tile that is exactly 2^E times e4m3 values splits into
    hi = those values and lo = 0."""
    rng = np.random.default_rng(6)
    codes = _codes(rng, (2, 128))
    codes[:, 0] = 0x7E  # make 448 the tile maximum so E = 0 after scaling by 2^3
    v = of.decode(codes) * 8.0
    E, hi, lo = of.split_activations(v)
    assert np.all(E == 3) and np.array_equal(hi * 8.0, v) and not lo.any()
