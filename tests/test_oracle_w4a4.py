"""Pins of the oracle's MXFP4 activation quantization and W4A4 GEMM (CPU).

The quantization restates the OCP Microscaling conversion: per block of 32, shared exponent
floor(log2 amax) - 2 (e2m1's largest exponent) as E8M0, elements rounded to nearest even
on the e2m1 grid with saturation.  Each pin checks it against something else: a
nearest-value search over the e2m1 grid, hand-worked blocks, an invariance, an error bound
and a rational brute force of the GEMM.
"""
from fractions import Fraction

import numpy as np

import oracle
from oracle import formats as F
from tests.conftest import load_golden
import workloads as WL

_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]          # e2m1 magnitudes, codes 0..7


def _nearest_e2m1(v):
    """Nearest e2m1 value by search; ties to the code with an even last bit; beyond 6: 6."""
    best = None
    for code, g in enumerate(_GRID):
        d = abs(abs(v) - g)
        if best is None or d < best[0] or (d == best[0] and code % 2 == 0):
            best = (d, code, g)
    return float(np.copysign(best[2], v))


def test_e2m1_rounding_matches_nearest_search():
    r = np.random.Generator(np.random.PCG64(3))
    vals = np.concatenate([np.arange(-9 * 64, 9 * 64 + 1) / 64.0, r.uniform(-10, 10, 2000)])
    got = F.round_to_e2m1_satfinite(vals)
    want = np.array([_nearest_e2m1(v) for v in vals])
    np.testing.assert_array_equal(got, want)
    # every grid value encodes to its code, -0 to 8
    np.testing.assert_array_equal(F.e2m1_encode(np.array(_GRID)), np.arange(8))
    np.testing.assert_array_equal(F.e2m1_encode(-np.array(_GRID[1:])), np.arange(9, 16))
    assert F.e2m1_encode(np.array([-0.0]))[0] == 8


def _block(vals):
    x = np.zeros((1, 32))
    x[0, :len(vals)] = vals
    return F.float_to_bf16_bits(x)


def _quant(vals):
    codes, e = oracle.quant_act_mxfp4(_block(vals))
    return oracle.unpack_nibbles(codes)[0], int(e[0, 0])


def test_mxfp4_quant_worked_blocks():
    # all ones: floor(log2 1) - 2 = -2 -> E8M0 125, elements 1 / 2^-2 = 4 (code 6)
    q, e = _quant([1.0] * 32)
    assert e == 125 and np.all(q == 6)
    # amax 7: exponent 2 - 2 = 0 -> E8M0 127; 7 saturates to 6 (code 7)
    q, e = _quant([7.0, 1.0])
    assert e == 127 and q[0] == 7 and q[1] == 2
    # amax 6 * 2^-5: exponent -3 - 2 = -5 -> 122; 6 and 3 after scaling (codes 7, 5)
    q, e = _quant([6.0 * 2 ** -5, 3.0 * 2 ** -5, -1.5 * 2 ** -5])
    assert e == 122 and list(q[:3]) == [7, 5, 11]
    # ties to even on the scaled values: amax 4 -> 127; 2.5 -> 2, -5 -> -4, 0.25 -> 0
    q, e = _quant([4.0, 2.5, -5.0, 0.25])
    assert e == 127 and list(q[:4]) == [6, 4, 14, 0]
    # an all-zero block: scale 1 (E8M0 127), zero codes
    q, e = _quant([])
    assert e == 127 and np.all(q == 0)


def test_mxfp4_quant_power_of_two_invariance():
    x = WL.gen_x(np.random.Generator(np.random.PCG64(4)), 4, 128)
    c0, e0 = oracle.quant_act_mxfp4(x)
    for j in (-3, 1, 5):
        xs = F.float_to_bf16_bits(F.bf16_bits_to_float(x) * 2.0 ** j)
        c, e = oracle.quant_act_mxfp4(xs)
        np.testing.assert_array_equal(c, c0)
        np.testing.assert_array_equal(e.astype(int), e0.astype(int) + j)


def test_mxfp4_quant_error_bound():
    """Rounding moves an element by at most half a spacing (1 x 2^s in the top binade), and
    saturation by less than 2 x 2^s (amax < 8 x 2^s), s = E - 127."""
    x = WL.gen_x(np.random.Generator(np.random.PCG64(5)), 8, 256, outliers=True)
    codes, e = oracle.quant_act_mxfp4(x)
    err = np.abs(oracle.dequant_act_mxfp4(codes, e) - F.bf16_bits_to_float(x))
    bound = np.ldexp(2.0, e.astype(np.int64) - 127)[:, np.arange(256) // 32]
    assert np.all(err <= bound)


def test_w4a4_rational_brute_force():
    tab = {int(k): Fraction(v[0][0]) for k, v in load_golden("e2m1_table.txt").items()}
    r = np.random.Generator(np.random.PCG64(6))
    M, N, K = 2, 3, 64
    xc = r.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    xe = r.integers(120, 134, size=(M, K // 32), dtype=np.uint8)
    wc = r.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    we = r.integers(120, 134, size=(N, K // 32), dtype=np.uint8)
    y = oracle.w4a4(xc, xe, "mxfp4", 32, wc, we)

    def val(codes, exps, row, k):
        byte = int(codes[row, k // 2])
        nib = (byte >> 4) if k % 2 else (byte & 15)
        return tab[nib] * Fraction(2) ** (int(exps[row, k // 32]) - 127)

    for m in range(M):
        for n in range(N):
            want = sum(val(xc, xe, m, k) * val(wc, we, n, k) for k in range(K))
            assert Fraction(y[m, n]) == want, (m, n)


def test_w4a4_of_quantized_activations_is_close():
    """End to end on the oracle: W4A4 on quantized X approximates the BF16 product within
    the activation rounding (a loose sanity check of the composition)."""
    r = np.random.Generator(np.random.PCG64(7))
    x = WL.gen_x(r, 4, 256)
    w = WL.gen_weights(r, "mxfp4", 16, 256)
    xq, xe = oracle.quant_act_mxfp4(x)
    y4 = oracle.w4a4(xq, xe, w.wfmt, w.group, w.codes, w.scales)
    y16 = oracle.w4a16(x, w.wfmt, w.group, w.codes, w.scales)
    rel = np.linalg.norm(y4 - y16) / np.linalg.norm(y16)
    assert rel < 0.2
