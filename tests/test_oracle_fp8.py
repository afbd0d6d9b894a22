"""Pins of the oracle's FP8 E4M3 quantiser against the format's definition
(landmark codes and values worked out by hand), brute force over every
finite code, and torch's float8_e4m3fn cast; plus the scale handling."""

import numpy as np
import pytest

from oracle import fp8


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x38, 1.0), (0x30, 0.5), (0x40, 2.0), (0xC0, -2.0), (0x3C, 1.5),
    (0x7E, 448.0), (0xFE, -448.0), (0x08, 2.0 ** -6), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9),
    (0x77, 240.0), (0x78, 256.0),
])
def test_landmark_codes(code, value):
    # 0x38 = 0 0111 000: e = 7 -> 2^0; 0x7E = 0 1111 110: 2^8 * 1.75 = 448;
    # 0x01: subnormal 2^-6 * 1/8; 0x77 = 0 1110 111: 2^7 * 1.875 = 240.
    assert fp8.decode([code])[0] == value
    assert fp8.encode([value])[0] == code


def test_nan_codes_and_count_of_finite_values():
    v = fp8.CODE_VALUES
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.isfinite(v).sum() == 254
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)                      # codes 0..0x7E increase


@pytest.mark.parametrize("y,code", [
    (1.0625, 0x38),      # halfway 1.0 (m=000) / 1.125 (m=001): even -> 1.0
    (1.1875, 0x3A),      # halfway 1.125 (001) / 1.25 (010): even -> 1.25
    (1.07, 0x39),        # nearer 1.125
    (2.0 ** -10, 0x00),  # halfway 0 / 2^-9: even -> 0
    (3 * 2.0 ** -10, 0x02),   # halfway 2^-9 (code 1) / 2^-8 (code 2): even -> code 2
    (-(2.0 ** -11), 0x80),    # rounds to zero, keeps the sign
    (464.0, 0x7E),       # beyond 448 saturates
    (1e6, 0x7E), (-1e6, 0xFE),
    (0.0, 0x00), (-0.0, 0x80),
])
def test_rounding_ties_subnormals_saturation(y, code):
    assert fp8.encode([y])[0] == code


def test_encode_is_nearest_by_brute_force():
    rng = np.random.default_rng(0)
    y = np.concatenate([rng.standard_normal(4000) * 3, rng.uniform(-460, 460, 2000),
                        rng.uniform(-0.02, 0.02, 2000)]).astype(np.float32)
    codes = fp8.encode(y)
    finite = [c for c in range(256) if np.isfinite(fp8.CODE_VALUES[c])]
    vals = fp8.CODE_VALUES[finite]
    for yi, ci in zip(y.astype(np.float64), codes):
        a = min(abs(yi), 448.0) * (1 if yi >= 0 else -1)
        d = np.abs(vals - a)
        best = d.min()
        cands = [finite[i] for i in np.nonzero(d == best)[0]]
        cands = [c for c in cands if (c & 0x80) == (0x80 if yi < 0 else 0)] or cands
        if len(cands) > 1:                               # a tie: the even code
            cands = [c for c in cands if c % 2 == 0]
        assert ci in cands, (yi, ci, cands)


def test_encode_matches_torch_float8_cast_in_range():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn")
    rng = np.random.default_rng(1)
    y = np.concatenate([rng.standard_normal(20000) * 4, rng.uniform(-448, 448, 5000),
                        rng.uniform(-0.05, 0.05, 5000)]).astype(np.float32)
    want = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(fp8.encode(y), want)


def test_quantize_uses_fp32_reciprocal_scale():
    # x * fp32(1/3) differs from x / 3 in the last fp32 place for some x;
    # the quantiser follows the multiply.
    x = np.array([1.5, -0.75, 3.0, 0.1], dtype=np.float16)
    inv = np.float32(1.0) / np.float32(3.0)
    np.testing.assert_array_equal(fp8.quantize(x, 3.0), fp8.encode(x.astype(np.float32) * inv))
    np.testing.assert_allclose(fp8.dequantize(fp8.quantize(x, 3.0), 3.0),
                               fp8.decode(fp8.quantize(x, 3.0)) * 3.0, rtol=0, atol=0)
    # scale 1: quantise-then-dequantise of an exactly representable value is exact
    exact = np.array([1.0, -2.5, 448.0, 2.0 ** -9], dtype=np.float16)
    np.testing.assert_array_equal(fp8.dequantize(fp8.quantize(exact, 1.0), 1.0), exact.astype(np.float64))


def test_relative_error_bound_of_normals():
    # 3 mantissa bits: relative rounding error at most 2^-4 for normal values
    rng = np.random.default_rng(2)
    y = rng.uniform(2.0 ** -6, 448, 20000).astype(np.float32)
    rel = np.abs(fp8.decode(fp8.encode(y)) - y) / y
    assert rel.max() <= 2.0 ** -4 + 1e-12
