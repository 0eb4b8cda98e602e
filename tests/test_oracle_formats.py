"""Pins of the oracle's number formats against printed values and library routines."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from tests.conftest import load_golden


def test_e2m1_matches_printed_grid():
    g = load_golden("e2m1_table.txt")
    # the table lines are 'code value'; keys are the codes
    table = {int(k): v[0][0] for k, v in g.items()}
    assert sorted(table) == list(range(16))
    got = F.e2m1_to_float(np.arange(16))
    for c in range(16):
        assert got[c] == table[c], c
        assert np.signbit(got[c]) == np.signbit(table[c]), c


def test_e8m0_matches_torch():
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("torch has no float8_e8m0fnu")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = F.e8m0_to_float(codes)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = F.e4m3_to_float(codes)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])
    np.testing.assert_array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))
    assert got[0x7E] == 448.0 and np.isnan(got[0x7F])


def test_int4_signed_matches_arithmetic_shift():
    n = np.arange(16, dtype=np.int8)
    ref = (n << 4).astype(np.int8) >> 4          # sign extension by the integer unit
    np.testing.assert_array_equal(F.int4_signed(n), ref.astype(np.int64))


def _fp32_samples(r, n):
    a = r.standard_normal(n).astype(np.float32) * np.float32(3.0)
    b = np.ldexp(r.uniform(1, 2, n), r.integers(-140, 128, n)).astype(np.float32)
    # exact ties between neighbouring bf16 values
    base = torch.from_numpy(r.standard_normal(n).astype(np.float32)).to(torch.bfloat16)
    bits = base.view(torch.int16).numpy().astype(np.int64) & 0xFFFF
    tie = ((bits << 16) | 0x8000).astype(np.uint32).view(np.float32)
    special = np.array([0.0, -0.0, 1e-45, -1e-45, 3.4e38, -3.4e38, 3.3895e38, 3.39e38,
                        1.1754944e-38, 9.2e-41], dtype=np.float32)
    return np.concatenate([a, b, tie, special])


def test_round_to_bf16_matches_torch():
    r = np.random.Generator(np.random.PCG64(1))
    x = _fp32_samples(r, 20000)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = F.round_to_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(np.signbit(got), np.signbit(ref))


def test_round_to_bf16_overflow_and_bits():
    assert F.round_to_bf16(np.array([1e39]))[0] == np.inf
    assert F.round_to_bf16(np.array([F.BF16_MAX]))[0] == F.BF16_MAX
    v = np.array([1.0, -2.0, 0.5, 6.0, 2.0 ** -133])
    bits = F.float_to_bf16_bits(v)
    np.testing.assert_array_equal(F.bf16_bits_to_float(bits), v)
    assert list(bits[:3]) == [0x3F80, 0xC000, 0x3F00]


def test_round_to_e4m3_matches_torch_in_range():
    r = np.random.Generator(np.random.PCG64(2))
    x = np.concatenate([
        r.uniform(-464, 464, 20000), r.standard_normal(20000) * 0.01,
        np.ldexp(r.uniform(-2, 2, 5000), -9),
        F.e4m3_to_float(np.arange(0x7E)) + np.ldexp(1.0, -12),   # just above grid points
    ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = F.round_to_e4m3_satfinite(x.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_e4m3_saturation_and_encode():
    got = F.round_to_e4m3_satfinite(np.array([470.0, 1e6, -1e6, 449.0]))
    np.testing.assert_array_equal(got, [448.0, 448.0, -448.0, 448.0])
    vals = F.e4m3_to_float(np.arange(256))
    ok = ~np.isnan(vals)
    codes = F.e4m3_encode(vals[ok])
    np.testing.assert_array_equal(codes, np.arange(256)[ok])
