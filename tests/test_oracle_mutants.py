"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins catch each.

A pin set that lets a dropped term, a wrong sign, a wrong index or a transposed operand
through would not pin anything; every mutant below must make at least one pin fail.
"""
import numpy as np
import pytest

import oracle
from oracle import formats as F
from oracle import qgemm_oracle as Q
from tests import test_oracle_formats as TF
from tests import test_oracle_gemm as TG
from tests import test_oracle_w4a4 as TW

PINS = [
    TF.test_e2m1_matches_printed_grid, TF.test_e8m0_matches_torch,
    TF.test_e4m3_decode_matches_torch, TF.test_int4_signed_matches_arithmetic_shift,
    TF.test_round_to_bf16_matches_torch, TF.test_round_to_e4m3_matches_torch_in_range,
    lambda: TG.test_worked_int4_examples("worked_uint4_zp.txt"),
    lambda: TG.test_worked_int4_examples("worked_int4_sym.txt"),
    TG.test_worked_mxfp4_example, TG.test_nibble_order_low_is_even,
    TG.test_worked_bf16_weight_rounding,
    lambda: TG.test_integer_brute_force("int4_sym", 32),
    lambda: TG.test_integer_brute_force("uint4_zp", 64),
    lambda: TG.test_integer_brute_force("mxfp4", 32),
    TG.test_one_hot_reproduces_weight_columns, TG.test_zero_point_invariants,
    lambda: TG.test_group_boundary_selects_next_scale("uint4_zp", 128),
    lambda: TG.test_group_boundary_selects_next_scale("mxfp4", 32),
    TG.test_fp8_activation_worked_example, TG.test_fp8_activation_invariants,
    TG.test_w4a8_equals_dense_on_dequantized_activations, TG.test_moe_decomposition,
    lambda: TG.test_integer_brute_force("mxint4", 32),
    lambda: TG.test_integer_brute_force("nvfp4", 16),
    lambda: TG.test_group_boundary_selects_next_scale("nvfp4", 16),
    TG.test_worked_mxint4_and_nvfp4_values, TG.test_nvfp4_global_scale_multiplies_the_output,
    TW.test_e2m1_rounding_matches_nearest_search, TW.test_mxfp4_quant_worked_blocks,
    TW.test_mxfp4_quant_power_of_two_invariance, TW.test_mxfp4_quant_error_bound,
    TW.test_w4a4_rational_brute_force, TG.test_bias_is_added_after_the_scales,
]


def _some_pin_fails():
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            return True
    return False


def _unpack_swapped(codes):
    codes = np.asarray(codes, dtype=np.uint8)
    out = np.empty((codes.shape[0], 2 * codes.shape[1]), dtype=np.uint8)
    out[:, 0::2] = codes >> 4
    out[:, 1::2] = codes & 0xF
    return out


def _e2m1_bad_bias(codes):
    c = np.asarray(codes).astype(np.int64) & 0xF
    e, m = (c >> 1) & 3, c & 1
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + 0.5 * m, e))
    return np.where((c >> 3) & 1, -mag, mag)


def _e8m0_bad_bias(e):
    return np.ldexp(1.0, np.asarray(e).astype(np.int64) - 128)


def _int4_unsigned(n):
    return np.asarray(n).astype(np.int64) & 0xF


def _dequant_zp_sign(wfmt, group, codes, scales, zeros=None):
    if wfmt != "uint4_zp":
        return _orig_dequant(wfmt, group, codes, scales, zeros)
    q = Q.unpack_nibbles(codes).astype(np.int64)
    g = np.arange(q.shape[1]) // group
    return (q + zeros.astype(np.int64)[:, g]) * Q.scale_values(wfmt, scales)[:, g]


def _dequant_group_shift(wfmt, group, codes, scales, zeros=None):
    q = Q.unpack_nibbles(codes)
    k = q.shape[1]
    g = np.minimum((np.arange(k) + 1) // group, k // group - 1)   # off by one position
    s = Q.scale_values(wfmt, scales)[:, g]
    if wfmt == "int4_sym":
        return F.int4_signed(q) * s
    if wfmt == "uint4_zp":
        return (q.astype(np.int64) - zeros.astype(np.int64)[:, g]) * s
    return F.e2m1_to_float(q) * s


def _gemm_transposed(x, w, chan_scale=None, tok_scale=None, bias=None):
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    y = x @ w.T[:, ::-1] if w.shape[0] > 1 else x @ w.T        # columns in reverse order
    if tok_scale is not None:
        y = y * np.asarray(tok_scale, dtype=np.float64)[:, None]
    return y


def _w4a16_bf16_weights(x_bits, wfmt, group, codes, scales, zeros=None, chan_scale=None,
                        global_scale=1.0):
    x = F.bf16_bits_to_float(x_bits)
    w = F.round_to_bf16(Q.dequant(wfmt, group, codes, scales, zeros))
    return Q.gemm(x, w, chan_scale=chan_scale) * np.float64(np.float32(global_scale))


def _gemm_drop_tok_scale(x, w, chan_scale=None, tok_scale=None, bias=None):
    return _orig_gemm(x, w, chan_scale=chan_scale, tok_scale=None, bias=bias)


def _quant_no_zero_guard(x_bits):
    x = F.bf16_bits_to_float(x_bits).astype(np.float32)
    amax = np.max(np.abs(x), axis=1)
    s = (amax / np.float32(448.0)).astype(np.float32)
    v = np.nan_to_num(x / s[:, None])
    return F.e4m3_encode(F.round_to_e4m3_satfinite(v.astype(np.float64))), s


def _scale_values_nvfp4_as_e8m0(wfmt, scales):
    if wfmt == "nvfp4":
        return F.e8m0_to_float(scales)
    return _orig_scale_values(wfmt, scales)


def _dequant_mxint4_as_e2m1(wfmt, group, codes, scales, zeros=None, global_scale=1.0):
    if wfmt == "mxint4":
        wfmt = "mxfp4"
    return _orig_dequant(wfmt, group, codes, scales, zeros, global_scale)


def _dequant_global_dropped(wfmt, group, codes, scales, zeros=None, global_scale=1.0):
    return _orig_dequant(wfmt, group, codes, scales, zeros)


def _e2m1_ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    q = np.ldexp(1.0, np.maximum(e, 1) - 2)
    r = np.sign(x) * np.floor(np.abs(x) / q + 0.5) * q
    return np.clip(r, -6.0, 6.0)


def _quant_act_mxfp4_exp_minus_one(x_bits, block=32):
    x = F.bf16_bits_to_float(x_bits)
    m, k = x.shape
    xb = x.reshape(m, k // block, block)
    amax = np.max(np.abs(xb), axis=2)
    _, e2 = np.frexp(amax)
    e = np.clip(np.where(amax > 0, (e2 - 1) - 1 + 127, 127), 0, 254).astype(np.int64)
    q = F.round_to_e2m1_satfinite(xb / np.ldexp(1.0, e - 127)[..., None])
    nib = F.e2m1_encode(q).reshape(m, k)
    return (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8), e.astype(np.uint8)


def _dequant_act_block_shifted(codes, exps, block=32):
    q = Q.unpack_nibbles(codes)
    k = q.shape[1]
    g = np.minimum((np.arange(k) + 1) // block, k // block - 1)
    return F.e2m1_to_float(q) * F.e8m0_to_float(exps)[:, g]


def _gemm_bias_scaled(x, w, chan_scale=None, tok_scale=None, bias=None):
    y = np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64)[None, :]
    if tok_scale is not None:
        y = y * np.asarray(tok_scale, dtype=np.float64)[:, None]
    if chan_scale is not None:
        y = y * np.asarray(chan_scale, dtype=np.float64)[None, :]
    return y


_orig_dequant = Q.dequant
_orig_gemm = Q.gemm
_orig_scale_values = Q.scale_values

MUTANTS = {
    "nibble order swapped": (Q, "unpack_nibbles", _unpack_swapped),
    "e2m1 exponent bias": (F, "e2m1_to_float", _e2m1_bad_bias),
    "e8m0 bias 128": (F, "e8m0_to_float", _e8m0_bad_bias),
    "int4 read unsigned": (F, "int4_signed", _int4_unsigned),
    "zero point added": (Q, "dequant", _dequant_zp_sign),
    "group index shifted": (Q, "dequant", _dequant_group_shift),
    "output columns permuted": (Q, "gemm", _gemm_transposed),
    "token scale dropped": (Q, "gemm", _gemm_drop_tok_scale),
    "w4a16 on bf16-rounded weights": (Q, "w4a16", _w4a16_bf16_weights),
    "zero row not guarded": (Q, "quant_act_fp8", _quant_no_zero_guard),
    "nvfp4 scale read as e8m0": (Q, "scale_values", _scale_values_nvfp4_as_e8m0),
    "mxint4 read as e2m1": (Q, "dequant", _dequant_mxint4_as_e2m1),
    "global scale dropped": (Q, "dequant", _dequant_global_dropped),
    "e2m1 ties away from zero": (F, "round_to_e2m1_satfinite", _e2m1_ties_away),
    "mxfp4 act exponent minus one": (Q, "quant_act_mxfp4", _quant_act_mxfp4_exp_minus_one),
    "act block index shifted": (Q, "dequant_act_mxfp4", _dequant_act_block_shifted),
    "bias added before the scales": (Q, "gemm", _gemm_bias_scaled),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    mod, attr, fn = MUTANTS[name]
    monkeypatch.setattr(mod, attr, fn)
    # the package-level re-exports must see the mutant too
    if hasattr(oracle, attr) and mod is Q:
        monkeypatch.setattr(oracle, attr, fn)
    with np.errstate(all="ignore"):
        assert _some_pin_fails(), f"no pin caught: {name}"


def test_unmutated_oracle_passes_every_pin():
    assert not _some_pin_fails()
