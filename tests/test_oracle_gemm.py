"""Pins of the oracle's dequantization, GEMM, FP8 activation quantization and MoE path.

Each test checks the oracle against something other than itself: hand-worked examples,
brute force with integer/rational arithmetic, closed-form invariants and decompositions.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import formats as F
from tests.conftest import load_golden
import workloads as WL


def _golden_weights(name):
    g = load_golden(name)
    N, K, group = g["N"][0][0], g["K"][0][0], g["group"][0][0]
    wfmt = g["wfmt"][0][0]
    codes = np.array(g["codes"], dtype=np.uint8).reshape(N, K // 2)
    sdt = np.uint8 if wfmt == "mxfp4" else np.uint16
    scales = np.array(g["scales"], dtype=sdt).reshape(N, K // group)
    zeros = np.array(g["zeros"], dtype=np.uint8).reshape(N, K // group) if "zeros" in g else None
    return g, wfmt, group, codes, scales, zeros


@pytest.mark.parametrize("name", ["worked_uint4_zp.txt", "worked_int4_sym.txt"])
def test_worked_int4_examples(name):
    g, wfmt, group, codes, scales, zeros = _golden_weights(name)
    W = oracle.dequant(wfmt, group, codes, scales, zeros)
    np.testing.assert_array_equal(W, np.array(g["W"], dtype=np.float64))
    X = np.array(g["X"], dtype=np.float64)
    xb = F.float_to_bf16_bits(X)
    Y = oracle.w4a16(xb, wfmt, group, codes, scales, zeros)
    np.testing.assert_array_equal(Y, np.array(g["Y"], dtype=np.float64))


def test_worked_bf16_weight_rounding():
    g, wfmt, group, codes, scales, zeros = _golden_weights("worked_bf16_weights.txt")
    np.testing.assert_array_equal(oracle.dequant(wfmt, group, codes, scales, zeros),
                                  np.array(g["Wexact"], dtype=np.float64))
    np.testing.assert_array_equal(oracle.dequant_bf16(wfmt, group, codes, scales, zeros),
                                  np.array(g["W"], dtype=np.float64))
    xb = F.float_to_bf16_bits(np.array(g["X"], dtype=np.float64))
    Y = oracle.w4a16(xb, wfmt, group, codes, scales, zeros)
    np.testing.assert_array_equal(Y, np.array(g["Y"], dtype=np.float64))


def test_worked_mxfp4_example():
    g, wfmt, group, codes, scales, zeros = _golden_weights("worked_mxfp4.txt")
    W = oracle.dequant(wfmt, group, codes, scales)
    expect = np.zeros((1, 64))
    for k, v in g["Wnz"][0]:
        expect[0, k] = v
    np.testing.assert_array_equal(W, expect)
    assert np.signbit(W[0, 3])                              # code 8 is -0
    xb = F.float_to_bf16_bits(np.ones((1, 64)))
    Y = oracle.w4a16(xb, wfmt, group, codes, scales)
    assert Y[0, 0] == g["Y"][0][0]


def test_nibble_order_low_is_even():
    codes = np.array([[0x21, 0x43]], dtype=np.uint8)
    np.testing.assert_array_equal(oracle.unpack_nibbles(codes), [[1, 2, 3, 4]])


# --- brute force on tiny integer-valued inputs ------------------------------------------

def _e2m1_table():
    g = load_golden("e2m1_table.txt")
    return {int(k): Fraction(v[0][0]) for k, v in g.items()}


def _e4m3_fraction(code):
    """E4M3 (OCP "fn") code -> exact rational, from the format definition: exponent field
    e (bias 7), mantissa m, value (1 + m/8) 2^(e-7), or m/8 2^-6 when e == 0."""
    e, m = (code >> 3) & 15, code & 7
    v = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return -v if code & 0x80 else v


def _brute_force(wfmt, group, codes, scales_val, zeros, x_int, g=Fraction(1)):
    """y[m][n] with Python rationals: nibble k from byte k//2 (low nibble for even k)."""
    tab = _e2m1_table()
    N, Kh = codes.shape
    K = 2 * Kh
    M = len(x_int)
    y = [[Fraction(0)] * N for _ in range(M)]
    for n in range(N):
        for k in range(K):
            byte = int(codes[n, k // 2])
            nib = (byte >> 4) if (k % 2) else (byte & 15)
            s = scales_val[n][k // group]
            if wfmt in ("int4_sym", "mxint4"):
                w = (nib - 16 if nib >= 8 else nib) * s
            elif wfmt == "uint4_zp":
                w = (nib - int(zeros[n, k // group])) * s
            else:
                w = tab[nib] * s
            for m in range(M):
                y[m][n] += x_int[m][k] * w * g
    return y


@pytest.mark.parametrize("wfmt,group", [("int4_sym", 32), ("uint4_zp", 64), ("mxfp4", 32),
                                        ("mxint4", 32), ("nvfp4", 16)])
def test_integer_brute_force(wfmt, group):
    r = np.random.Generator(np.random.PCG64(7))
    M, N, K = 3, 5, 128
    x_int = r.integers(-4, 5, size=(M, K))
    codes = r.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    G = K // group
    g, gf = 1.0, Fraction(1)
    if wfmt in ("mxfp4", "mxint4"):
        exps = r.integers(124, 131, size=(N, G), dtype=np.uint8)
        scales = exps
        scales_val = [[Fraction(2) ** (int(e) - 127) for e in row] for row in exps]
        zeros = None
    elif wfmt == "nvfp4":
        # every E4M3 code but NaN, subnormals included, either sign; a float32 global scale
        scales = r.integers(0, 256, size=(N, G), dtype=np.uint8)
        scales[(scales & 0x7F) == 0x7F] = 0x38
        scales_val = [[_e4m3_fraction(int(c)) for c in row] for row in scales]
        zeros = None
        g = float(np.float32(0.3))
        gf = Fraction(g)
    else:
        p = r.integers(-3, 3, size=(N, G))
        sv = np.ldexp(1.0, p)
        scales = F.float_to_bf16_bits(sv)
        scales_val = [[Fraction(2) ** int(e) for e in row] for row in p]
        zeros = r.integers(0, 16, size=(N, G), dtype=np.uint8) if wfmt == "uint4_zp" else None
    xb = F.float_to_bf16_bits(x_int.astype(np.float64))
    Y = oracle.w4a16(xb, wfmt, group, codes, scales, zeros, global_scale=g)
    ref = _brute_force(wfmt, group, codes, scales_val, zeros, x_int.tolist(), gf)
    for m in range(M):
        for n in range(N):
            assert Fraction(Y[m, n]) == ref[m][n], (m, n)


def test_one_hot_reproduces_weight_columns():
    x, w = WL.tiny_dense(seed=3)
    W = oracle.dequant(w.wfmt, w.group, w.codes, w.scales, w.zeros)
    # the scales of this workload make most weights need more than BF16's 8 bits
    assert np.any(W != oracle.dequant_bf16(w.wfmt, w.group, w.codes, w.scales, w.zeros))
    K = w.K
    for k in (0, 1, 127, 128, 129, K - 1):
        onehot = np.zeros((1, K))
        onehot[0, k] = 1.0
        y = oracle.w4a16(F.float_to_bf16_bits(onehot), w.wfmt, w.group, w.codes, w.scales)
        np.testing.assert_array_equal(y[0], W[:, k])


def test_zero_point_invariants():
    r = np.random.Generator(np.random.PCG64(5))
    N, K, g = 16, 256, 128
    nib = r.integers(0, 16, size=(N, K), dtype=np.uint8)
    codes = WL.pack_nibbles(nib)
    s = WL.to_bf16_bits(r.uniform(0.005, 0.02, size=(N, K // g)).astype(np.float32))
    # a two's-complement nibble n has value (n xor 8) - 8: uint4 with z = 8 on n ^ 8
    sym = oracle.dequant("int4_sym", g, codes, s)
    asym = oracle.dequant("uint4_zp", g, WL.pack_nibbles(nib ^ 8), s,
                          np.full((N, K // g), 8, np.uint8))
    np.testing.assert_array_equal(sym, asym)
    # z equal to every code of its group -> all-zero weights
    const = np.repeat(r.integers(0, 16, size=(N, K // g), dtype=np.uint8), g, axis=1)
    w0 = oracle.dequant("uint4_zp", g, WL.pack_nibbles(const), s, const[:, ::g])
    assert np.all(w0 == 0)
    # a zero point moves the weight the other way from the code
    z1 = np.full((N, K // g), 1, np.uint8)
    z0 = np.zeros((N, K // g), np.uint8)
    d = oracle.dequant("uint4_zp", g, codes, s, z0) - oracle.dequant("uint4_zp", g, codes, s, z1)
    np.testing.assert_array_equal(d, F.bf16_bits_to_float(s)[:, np.arange(K) // g])


def test_scale_linearity():
    x, w = WL.tiny_dense(seed=4)
    y1 = oracle.w4a16(x, w.wfmt, w.group, w.codes, w.scales)
    s2 = (w.scales.astype(np.uint32) + (1 << 7)).astype(np.uint16)   # exponent + 1
    y2 = oracle.w4a16(x, w.wfmt, w.group, w.codes, s2)
    np.testing.assert_array_equal(y2, 2 * y1)
    xm, wm = WL.mxfp4_shape(64, 256, 4, seed=4)
    y1 = oracle.w4a16(xm, wm.wfmt, wm.group, wm.codes, wm.scales)
    y2 = oracle.w4a16(xm, wm.wfmt, wm.group, wm.codes, wm.scales + 1)
    np.testing.assert_array_equal(y2, 2 * y1)


@pytest.mark.parametrize("wfmt,group", [("uint4_zp", 128), ("mxfp4", 32), ("mxint4", 32),
                                        ("nvfp4", 16)])
def test_group_boundary_selects_next_scale(wfmt, group):
    r = np.random.Generator(np.random.PCG64(6))
    N, K = 8, 4 * group
    nib = np.full((N, K), 2, np.uint8)                    # int 2 / e2m1 1.0 everywhere
    codes = WL.pack_nibbles(nib)
    if wfmt in ("mxfp4", "mxint4"):
        scales = r.integers(100, 140, size=(N, K // group), dtype=np.uint8)
        zeros = None
        sv = np.ldexp(1.0, scales.astype(np.int64) - 127)
        unit = 1.0 if wfmt == "mxfp4" else 2.0
    elif wfmt == "nvfp4":
        scales = r.integers(0x08, 0x78, size=(N, K // group), dtype=np.uint8)   # normals
        zeros = None
        sv = np.array([[float(_e4m3_fraction(int(c))) for c in row] for row in scales])
        unit = 1.0
    else:
        scales = WL.to_bf16_bits(r.uniform(0.5, 2, size=(N, K // group)).astype(np.float32))
        zeros = np.zeros((N, K // group), np.uint8)
        sv = F.bf16_bits_to_float(scales)
        unit = 2.0
    W = oracle.dequant(wfmt, group, codes, scales, zeros)
    for j in range(K // group):
        np.testing.assert_array_equal(W[:, j * group], unit * sv[:, j])
        np.testing.assert_array_equal(W[:, j * group + group - 1], unit * sv[:, j])


def test_worked_mxint4_and_nvfp4_values():
    """Hand-worked weights from the format definitions.  MXINT4, E8M0 129 (x4): nibbles
    8, 7, 15, 1 are -8, 7, -1, 1 -> -32, 28, -4, 4.  NVFP4 with per-tensor scale 0.5:
    e2m1 7 (6.0) x E4M3 0x38 (1.0) -> 3.0; e2m1 11 (-1.5) x 0x01 (the smallest subnormal,
    2^-9) -> -1.5 * 2^-10; e2m1 1 (0.5) x 0x7E (448) -> 112; e2m1 8 (-0) x 0x50 (4.0) -> -0."""
    codes = np.array([[0x78, 0x1F] + [0] * 14], dtype=np.uint8)        # 32 elements
    W = oracle.dequant("mxint4", 32, codes, np.array([[129]], dtype=np.uint8))
    np.testing.assert_array_equal(W[0, :4], [-32.0, 28.0, -4.0, 4.0])
    for j, (c, sc, want) in enumerate([(7, 0x38, 3.0), (11, 0x01, -1.5 * 2.0 ** -10),
                                       (1, 0x7E, 112.0), (8, 0x50, -0.0)]):
        cd = np.zeros((1, 8), np.uint8)                                  # 16 elements
        cd[0, 0] = c
        w = oracle.dequant("nvfp4", 16, cd, np.array([[sc]], dtype=np.uint8), global_scale=0.5)
        assert w[0, 0] == want and np.signbit(w[0, 0]) == np.signbit(want), (j, w[0, 0])


def test_nvfp4_global_scale_multiplies_the_output():
    """The per-tensor scale multiplies the output, after the BF16 operand e2m1 x E4M3
    (exact): a one-hot row reproduces g x e2m1 x s without a BF16 rounding of the product
    with g, and y(g) = g y(1)."""
    r = np.random.Generator(np.random.PCG64(11))
    w = WL.gen_weights(r, "nvfp4", 6, 64)
    g = float(np.float32(0.1234567))
    exact = oracle.dequant("nvfp4", 16, w.codes, w.scales, global_scale=g)
    assert np.any(F.round_to_bf16(exact) != exact)           # g makes the product inexact
    for k in (0, 15, 16, 63):
        onehot = np.zeros((1, 64))
        onehot[0, k] = 1.0
        y = oracle.w4a16(F.float_to_bf16_bits(onehot), "nvfp4", 16, w.codes, w.scales,
                         global_scale=g)
        np.testing.assert_array_equal(y[0], exact[:, k])
    x = WL.gen_x(r, 3, 64)
    y1 = oracle.w4a16(x, "nvfp4", 16, w.codes, w.scales)
    yg = oracle.w4a16(x, "nvfp4", 16, w.codes, w.scales, global_scale=g)
    np.testing.assert_array_equal(yg, y1 * g)


def test_bias_is_added_after_the_scales():
    """Integer X, power-of-two weights, a dyadic bias: every step is exact, so the bias
    shows up unscaled on top of the scaled sum, once per output column."""
    r = np.random.Generator(np.random.PCG64(12))
    x = r.integers(-3, 4, size=(3, 64)).astype(np.float64)
    w = np.ldexp(1.0, r.integers(-2, 2, size=(5, 64)))
    c = np.array([0.5, 2.0, 1.0, 4.0, 0.25])
    t = np.array([2.0, 0.5, 1.0])
    b = np.array([0.125, -3.0, 0.0, 7.5, -0.25])
    y = oracle.gemm(x, w, chan_scale=c, tok_scale=t, bias=b)
    base = (x @ w.T) * t[:, None] * c[None, :]
    np.testing.assert_array_equal(y - base, np.broadcast_to(b, y.shape))
    np.testing.assert_array_equal(oracle.gemm(x, w, bias=b) - x @ w.T, np.broadcast_to(b, y.shape))


def test_fp8_activation_worked_example():
    g = load_golden("worked_fp8_act.txt")
    X = np.array(g["X"], dtype=np.float64)
    codes, s = oracle.quant_act_fp8(F.float_to_bf16_bits(X))
    np.testing.assert_array_equal(codes, np.array(g["codes"], dtype=np.uint8))
    assert s[0] == np.float32(100.0) / np.float32(448.0)
    assert s[1] == g["scale_row1"][0][0]


def test_fp8_activation_invariants():
    r = np.random.Generator(np.random.PCG64(8))
    xb = WL.gen_x(r, 32, 512, outliers=True)
    codes, s = oracle.quant_act_fp8(xb)
    x = F.bf16_bits_to_float(xb)
    amax_rows = np.argmax(np.abs(x), axis=1)
    top = codes[np.arange(32), amax_rows]
    assert np.all((top & 0x7F) == 0x7E)                  # the row maximum maps to +-448
    deq = F.e4m3_to_float(codes) * s[:, None].astype(np.float64)
    rel = np.abs(deq - x) / np.maximum(np.abs(x), 1e-30)
    big = np.abs(x) >= s[:, None] * 2.0 ** -6             # normal e4m3 range
    assert np.max(rel[big]) <= 2.0 ** -4 * 1.0001          # half an ulp of a 4-bit significand


def test_w4a8_equals_dense_on_dequantized_activations():
    xb, w = WL.mxfp4_shape(32, 256, 8, seed=9, outliers=True)
    codes, s = oracle.quant_act_fp8(xb)
    y = oracle.w4a8(codes, s, w.wfmt, w.group, w.codes, w.scales)
    W = oracle.dequant(w.wfmt, w.group, w.codes, w.scales)
    # brute force in rationals on a few entries
    xa = F.e4m3_to_float(codes)
    for (m, n) in [(0, 0), (3, 17), (7, 31)]:
        ref = sum(Fraction(xa[m, k]) * Fraction(W[n, k]) for k in range(256)) * Fraction(float(s[m]))
        assert abs(Fraction(y[m, n]) - ref) <= abs(ref) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 80)


def test_moe_decomposition():
    case = WL.moe_case(T=6, seed=1, E=4, topk=2, hidden=64, inter=32)
    ws = [WL.gen_weights(np.random.Generator(np.random.PCG64(e)), "mxfp4", 48, 64) for e in range(4)]
    Ws = [oracle.dequant(w.wfmt, w.group, w.codes, w.scales) for w in ws]
    x = F.bf16_bits_to_float(case.x_bits)
    y = oracle.moe_grouped(x, case.offsets, Ws)
    for e in range(4):
        a, b = case.offsets[e], case.offsets[e + 1]
        np.testing.assert_array_equal(y[a:b], x[a:b] @ Ws[e].T)
    # padding rows carry zero inputs and give zero outputs
    assert np.all(y[~case.valid] == 0)
    # one expert holding every row is the dense GEMM
    y1 = oracle.moe_grouped(x, np.array([0, x.shape[0]]), Ws[:1])
    np.testing.assert_array_equal(y1, oracle.gemm(x, Ws[0]))


def test_moe_indexed():
    """Gathering rows by index: equals the grouped GEMM on the rows sorted beforehand
    (including padding rows, which index -1 and give zeros), and does not depend on where
    the token rows lie (a permutation of x with the index remapped gives the same Y)."""
    case = WL.moe_case(T=9, seed=3, E=4, topk=2, hidden=64, inter=32)
    ws = [WL.gen_weights(np.random.Generator(np.random.PCG64(10 + e)), "int4_sym", 40, 64, group=32)
          for e in range(4)]
    Ws = [oracle.dequant(w.wfmt, w.group, w.codes, w.scales) for w in ws]
    x_tok = F.bf16_bits_to_float(case.x_tok_bits)
    x_sorted = F.bf16_bits_to_float(case.x_bits)
    y = oracle.moe_indexed(x_tok, case.offsets, case.token_of_row, Ws)
    ref = oracle.moe_grouped(x_sorted, case.offsets, Ws)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    assert np.all(y[case.token_of_row < 0] == 0) and np.any(case.token_of_row < 0)
    perm = np.random.Generator(np.random.PCG64(4)).permutation(case.T)
    inv = np.argsort(perm)                          # x_tok[t] now sits at row inv[t]
    idx = np.where(case.token_of_row >= 0, inv[np.maximum(case.token_of_row, 0)], -1)
    np.testing.assert_array_equal(oracle.moe_indexed(x_tok[perm], case.offsets, idx, Ws), y)
    # per-row token scales follow the gathered row
    s = np.linspace(0.5, 2.0, case.T)
    ys = oracle.moe_indexed(x_tok, case.offsets, case.token_of_row, Ws, tok_scale=s)
    rows = case.token_of_row >= 0
    np.testing.assert_allclose(ys[rows], y[rows] * s[case.token_of_row[rows]][:, None],
                               rtol=1e-12, atol=1e-12)


def test_routing_layout():
    case = WL.moe_case(T=50, seed=2, E=16, topk=4, hidden=32, inter=32)
    assert case.counts.sum() == 50 * 4
    assert np.all(np.diff(case.offsets) % WL.MOE_PAD == 0)
    for e in range(16):
        a = case.offsets[e]
        rows = case.token_of_row[a:a + case.counts[e]]
        assert np.all(np.diff(rows) > 0)                  # stable: token order kept
    x_tok = F.bf16_bits_to_float(case.x_bits)
    assert np.all(x_tok[~case.valid] == 0)


def test_tolerance_helper():
    ref = np.array([[1.0, -2.0, 0.0, 1e-6]])
    rms = np.sqrt(np.mean(ref ** 2))
    ok, worst = oracle.tolerance_ok(ref + 8e-3 * np.maximum(np.abs(ref), rms) * 0.99, ref, 8e-3)
    assert ok and worst < 1
    bad = ref.copy()
    bad[0, 2] += 8e-3 * rms * 1.5
    assert not oracle.tolerance_ok(bad, ref, 8e-3)[0]
    assert not oracle.tolerance_ok(ref * np.nan, ref, 8e-3)[0]


def test_tiny_dense_workload_shape():
    x, w = WL.tiny_dense(seed=0)
    assert x.shape == (16, 512) and w.codes.shape == (256, 256) and w.scales.shape == (256, 4)
    s = F.bf16_bits_to_float(w.scales)
    assert s.min() >= 0.0049 and s.max() <= 0.0201
