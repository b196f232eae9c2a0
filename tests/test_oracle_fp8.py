"""Pins of the oracle's FP8 E4M3 codec (CPU): the decoded value of every code
against torch's float8_e4m3fn conversion (a library routine), the format's
printed constants, round-to-nearest-even against torch on random values, the
exact round trip of every finite code, saturation and the sign of zero."""
import numpy as np
import pytest
import torch

from oracle import fp8


def test_every_code_decodes_like_torch():
    ours = fp8.decode(np.arange(256))
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.array_equal(np.signbit(ours[fin]), np.signbit(ref[fin]))


def test_format_constants():
    v = fp8.decode([0x00, 0x01, 0x07, 0x08, 0x38, 0x39, 0x7E, 0x80, 0xB8, 0xFE])
    assert v.tolist() == [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.125, 448.0, -0.0, -1.0, -448.0]
    assert np.isnan(fp8.decode([0x7F, 0xFF])).all()
    assert np.isnan(fp8.decode(np.arange(256))).sum() == 2


def test_finite_codes_round_trip():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(fp8.encode(fp8.decode(codes)), codes)


@pytest.mark.parametrize("seed", range(3))
def test_rounding_matches_torch_in_range(seed):
    rng = np.random.default_rng(seed)
    x = np.concatenate([rng.normal(0, s, 4000) for s in (1e-3, 1e-1, 1.0, 30.0)]).astype(np.float32)
    x = x[np.abs(x) <= fp8.MAX_FINITE]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.encode(x), ref)


def test_ties_go_to_the_even_code():
    # exact midpoints: between 1.0 (0x38) and 1.125 (0x39); between the two
    # smallest subnormals; between 0 and the smallest subnormal
    assert fp8.encode([1.0625, 3 * 2.0 ** -10, 2.0 ** -10, 1.1875]).tolist() == [0x38, 0x02, 0x00, 0x3A]


def test_saturation_nan_and_signed_zero():
    assert fp8.encode([500.0, -1e9, 448.0, 464.0]).tolist() == [0x7E, 0xFE, 0x7E, 0x7E]
    assert fp8.encode([np.nan]).tolist() == [0x7F]
    assert fp8.encode([0.0, -0.0]).tolist() == [0x00, 0x80]


def test_scaled_round_trip_error_bound():
    # relative error of a normal-range value is at most half an ulp: 2^-4
    rng = np.random.default_rng(7)
    x = rng.normal(0, 1, 10000)
    scale = 0.05
    y = fp8.dequantize(fp8.quantize(x, scale), scale)
    normal = np.abs(x / scale) >= 2.0 ** -6
    rel = np.abs(y[normal] - x[normal]) / np.abs(x[normal])
    assert rel.max() <= 2.0 ** -4 + 1e-12
