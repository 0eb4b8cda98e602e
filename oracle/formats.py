"""Number formats of the quantized GEMM, decoded and rounded the slow, obvious way.

TEST INFRASTRUCTURE ONLY. Nothing in the product package imports this module; only
tests/, __graft_entry__.smoke() and the CPU legs of bench.py do.

Sources. The pages on Humming name the formats but do not define them:
  * "蚂蚁与vLLM开源量化推理内核Humming" (aiproducthub.cn), paragraph 支持矩阵 (support
    matrix): FP8 (e4m3/e5m2), FP4 (e2m1), BF16 (e8m7), symmetric INT1-INT8 and INT1-INT8
    with dynamic zero points.
  * "Humming wird angekündigt" (vLLM blog, German edition), section "Eine einheitliche
    Quantisierungsdarstellung": weight format, scale granularity, scale dtype, zero
    points and secondary scales are separate parameters.
The bit-level meaning of each name is the public one: an "eXmY" float has one sign bit,
X exponent bits with bias 2^(X-1)-1, Y mantissa bits, and subnormals when the exponent
field is zero; E8M0 is the OCP Microscaling shared scale 2^(e-127) with e=255 meaning
NaN; FP8 e4m3 is the OCP "fn" variant (no infinities, S.1111.111 is NaN, max 448).

Every function works on numpy arrays and returns float64 (or integer codes).
"""
import numpy as np

__all__ = [
    "int4_signed", "e2m1_to_float", "e8m0_to_float", "e4m3_to_float", "bf16_bits_to_float",
    "round_to_bf16", "round_to_e4m3_satfinite", "e4m3_encode", "float_to_bf16_bits",
    "round_to_e2m1_satfinite", "e2m1_encode", "BF16_MAX", "E4M3_MAX", "E2M1_MAX",
]

BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127
E4M3_MAX = 448.0
E2M1_MAX = 6.0


def int4_signed(nibbles):
    """Two's-complement 4-bit value of each nibble (0..15 -> -8..7)."""
    n = np.asarray(nibbles).astype(np.int64) & 0xF
    return np.where(n >= 8, n - 16, n)


def e2m1_to_float(codes):
    """FP4 e2m1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.

    Exponent field 0 is subnormal: value = m * 2^(1-1) * 0.5.  Code 8 is -0.
    """
    c = np.asarray(codes).astype(np.int64) & 0xF
    sign = (c >> 3) & 1
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + 0.5 * m, e - 1))
    return np.where(sign == 1, -mag, mag)


def e8m0_to_float(e):
    """E8M0 shared scale: 2^(e-127); 255 encodes NaN."""
    e = np.asarray(e).astype(np.int64)
    return np.where(e == 255, np.nan, np.ldexp(1.0, e - 127))


def e4m3_to_float(codes):
    """FP8 e4m3 (fn): bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def bf16_bits_to_float(bits):
    """bfloat16 bit patterns (uint16) -> float64.  A bf16 is the top half of a binary32."""
    b = np.asarray(bits).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _round_binary(x, p, emin):
    """Round float64 values to the nearest number with p significant bits and minimum
    normal exponent emin (subnormals below 2^emin), ties to even.  No overflow handling."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                  # |x| = f * 2^e with 0.5 <= f < 1, so ulp = 2^(e-p)
    e = np.maximum(e, emin + 1)         # below 2^emin the spacing stays 2^(emin+1-p)
    q = np.ldexp(1.0, e - p)
    return np.round(x / q) * q          # np.round rounds halves to even


def round_to_bf16(x):
    """Round-to-nearest-even of float64 values to bfloat16 (8 significant bits, emin -126),
    overflowing to +-inf; returns float64 values on the bf16 grid."""
    r = _round_binary(x, 8, -126)
    return np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, r), r)


def float_to_bf16_bits(x):
    """bf16 bit patterns of values that are already on the bf16 grid (float64 in)."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def round_to_e4m3_satfinite(x):
    """Round-to-nearest-even to FP8 e4m3 (4 significant bits, emin -6), then clamp
    results beyond the largest finite value (448) to +-448 ("satfinite")."""
    r = _round_binary(x, 4, -6)
    return np.clip(r, -E4M3_MAX, E4M3_MAX)


def round_to_e2m1_satfinite(x):
    """Round-to-nearest-even to FP4 e2m1 (2 significant bits, emin 0, so spacing 0.5 below
    1), then clamp beyond the largest finite value (6) to +-6."""
    r = _round_binary(x, 2, 0)
    return np.clip(r, -E2M1_MAX, E2M1_MAX)


_E2M1_POS = e2m1_to_float(np.arange(8))          # codes 0..7, strictly increasing


def e2m1_encode(v):
    """Codes (0..15) of values already on the e2m1 grid (|v| <= 6); the sign bit (bit 3)
    follows the sign of v, so -0.0 encodes as 8."""
    v = np.asarray(v, dtype=np.float64)
    mag = np.abs(v)
    code = np.searchsorted(_E2M1_POS, mag).astype(np.int64)
    if not np.all(_E2M1_POS[np.minimum(code, 7)] == mag):
        raise ValueError("e2m1_encode: value not on the e2m1 grid")
    return (code | (np.signbit(v).astype(np.int64) << 3)).astype(np.uint8)


_E4M3_POS = e4m3_to_float(np.arange(0x7F))      # codes 0x00..0x7E, strictly increasing


def e4m3_encode(v):
    """Codes of values already on the e4m3 grid (|v| <= 448).  The sign bit follows the
    sign of v, so -0.0 encodes as 0x80."""
    v = np.asarray(v, dtype=np.float64)
    mag = np.abs(v)
    code = np.searchsorted(_E4M3_POS, mag).astype(np.int64)
    if not np.all(_E4M3_POS[np.minimum(code, 0x7E)] == mag):
        raise ValueError("e4m3_encode: value not on the e4m3 grid")
    return (code | (np.signbit(v).astype(np.int64) << 7)).astype(np.uint8)
