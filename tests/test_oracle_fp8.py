"""Pins of the oracle's FP8 (E4M3) quantiser (CPU only)."""
import numpy as np
import torch

from oracle import quant
from tests.conftest import golden


def test_decode_matches_specified_values():
    g = golden("ocp_e4m3_values.json")
    for code, val in g["codes"].items():
        got = quant.e4m3_decode([int(code, 16)])[0]
        assert got == val and np.signbit(got) == np.signbit(val), code
    for code in g["nan_codes"]:
        assert np.isnan(quant.e4m3_decode([int(code, 16)])[0])
    finite = quant.e4m3_decode(np.arange(0, 127, dtype=np.uint8))
    assert np.all(np.diff(finite) > 0) and finite[-1] == g["max_finite"]


def test_round_trip_of_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(quant.e4m3_encode(quant.e4m3_decode(codes)), codes)


def test_ties_go_to_even_and_large_values_saturate():
    assert quant.e4m3_encode([1.0625])[0] == 0x38        # between 1 (0x38) and 1.125 (0x39)
    assert quant.e4m3_encode([1.1875])[0] == 0x3A        # between 1.125 (0x39) and 1.25 (0x3A)
    assert quant.e4m3_encode([0.0009765625])[0] == 0x00  # half the smallest subnormal -> 0 (even)
    assert quant.e4m3_encode([1000.0, -1e9, 448.0, 464.0])[0] == 0x7E
    assert list(quant.e4m3_encode([-1e9, 464.0])) == [0xFE, 0x7E]
    assert quant.e4m3_encode([-1e-12])[0] == 0x80        # the sign survives rounding to zero


def test_matches_library_cast_in_range():
    """torch's float8_e4m3fn cast (round to nearest even) on values within +-448."""
    r = np.random.default_rng(4)
    x = np.concatenate([r.normal(scale=s, size=20000) for s in (0.003, 0.1, 1.0, 30.0, 150.0)])
    x = np.clip(x, -448, 448).astype(np.float32)
    want = torch.tensor(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(quant.e4m3_encode(x.astype(np.float64)), want)


def test_relative_error_bound_for_normals():
    r = np.random.default_rng(5)
    x = r.uniform(0.016, 440.0, size=50000) * r.choice([-1, 1], size=50000)
    err = np.abs(quant.e4m3_decode(quant.e4m3_encode(x)) - x) / np.abs(x)
    assert err.max() <= 2.0 ** -4 + 1e-15


def test_quantize_rows_uses_per_head_scales():
    x = np.array([[[2.0, -3.0], [2.0, -3.0]]], dtype=np.float32)      # [T=1, Hkv=2, D=2]
    codes = quant.quantize_rows(x, [1.0, 0.5])
    assert list(codes[0, 0]) == list(quant.e4m3_encode([2.0, -3.0]))
    assert list(codes[0, 1]) == list(quant.e4m3_encode([4.0, -6.0]))
    deq = quant.dequantize(codes, [1.0, 0.5], head_axis=1)
    assert np.array_equal(deq, x.astype(np.float64))
