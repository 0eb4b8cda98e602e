"""Plain CPU oracle of the quantized-weight GEMM  Y = X . dequant(Wq)^T.

TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and the CPU legs of
bench.py may import this module.  It shares no code, table or constant with the CUDA
library and never calls it.

What it computes, and where that comes from:
  * "Humming wird angekündigt" (vLLM blog, German edition), section "Eine einheitliche
    Quantisierungsdarstellung": a weight is described by its format, scale granularity
    (group size), scale dtype, zero points and secondary scales; activations have their own
    format.  Example given there: group-wise INT4 weights paired with BF16 activations.
  * Same page, sections "WnA16" and "W8A8 / W4A8 / W4A4": W4A16 (4-bit weights, BF16
    activations) and W4A8-MXFP4 (MXFP4 weights, FP8 activations), each dense and as an MoE
    grouped path; section "End-to-End-Inferenzleistung": FP8 activations are tokenwise.
  * "蚂蚁与vLLM开源量化推理内核Humming", paragraph 支持矩阵: symmetric INT weights and INT
    weights with zero points; FP4 e2m1 weights.
  * Same page, paragraph 架构设计 and the German page's "Gemeinsam genutzte
    CUDA-Komponenten": dequantization and scaling are fused into the GEMM and scaling can be
    fused into the output stage (the secondary per-channel scale below).

Readings where the pages are silent (each is listed in the design notes):
  * canonical codes: uint8 [N, K/2], element k of row n in byte k//2, even k in the low
    nibble;
  * INT4 symmetric: the nibble is a two's-complement q in [-8, 7], w = q * s[n, k//g];
  * INT4 with zero point: q, z in [0, 15], w = (q - z) * s[n, k//g] (no "+1" offset);
  * MXFP4: w = e2m1(q) * 2^(e[n, k//32] - 127);
  * MXINT4 (named beside NVFP4 for the B300 MoE results of the German page, section
    "WnA16"): the nibble is a two's-complement q in [-8, 7] with one E8M0 per 32 K,
    w = q * 2^(e[n, k//32] - 127) (no implicit fixed-point factor; one would only shift e);
  * NVFP4 (same place): w = e2m1(q) * e4m3(s[n, k//16]) * g with a float32 per-tensor g.
    The 16-bit operand is e2m1(q) * e4m3(s), which BF16 holds exactly, and g is a
    per-tensor secondary scale that multiplies the output (the output stage, as for the
    per-channel scale);
  * secondary scale: optional float32 c[n] multiplying output column n;
  * FP8 activation quantization: per row m, s_m = amax_m / 448 in float32 (1.0 when the row
    is all zero), codes = e4m3 round-to-nearest-even with saturation of x / s_m computed in
    float32.
  * MXFP4 activation quantization (for W4A4, section "W8A8 / W4A8 / W4A4": MX formats on
    Blackwell's tensor cores): the OCP Microscaling conversion restated -- per block of 32
    K-elements of a row, the shared exponent is floor(log2(amax)) minus e2m1's largest
    exponent (2), stored as E8M0 (clamped to 0..254; 127, i.e. 1, for an all-zero block),
    and each element is x / 2^(E-127) rounded to nearest even on the e2m1 grid with
    saturation at 6.

The matmul accumulates in float64 over the exact dequantized weights, for W4A16 and W4A8
alike; dequant_bf16 (the weights rounded to BF16) is what the bit-exact dequantization
check compares.  Nothing is blocked, fused or reordered beyond the plain definition.
"""
import numpy as np

from . import formats as F

WFMTS = ("int4_sym", "uint4_zp", "mxfp4", "mxint4", "nvfp4")


def unpack_nibbles(codes):
    """uint8 [N, K/2] -> uint8 [N, K] with element k taken from byte k//2, even k low."""
    codes = np.asarray(codes, dtype=np.uint8)
    n, kh = codes.shape
    out = np.empty((n, 2 * kh), dtype=np.uint8)
    out[:, 0::2] = codes & 0xF
    out[:, 1::2] = codes >> 4
    return out


def scale_values(wfmt, scales):
    """Per-group scale values as float64: BF16 bit patterns, E8M0 exponents (MXFP4, MXINT4)
    or E4M3 codes (NVFP4)."""
    if wfmt in ("mxfp4", "mxint4"):
        return F.e8m0_to_float(scales)
    if wfmt == "nvfp4":
        return F.e4m3_to_float(scales)
    return F.bf16_bits_to_float(scales)


def dequant(wfmt, group, codes, scales, zeros=None, global_scale=1.0):
    """Exact dequantized weights W [N, K] in float64.

    wfmt: "int4_sym" | "uint4_zp" | "mxfp4" | "mxint4" | "nvfp4"; group: K-elements per
    scale (32 for mxfp4 and mxint4, 16 for nvfp4); codes: uint8 [N, K/2]; scales: uint16
    bf16 bits [N, K/group], uint8 E8M0 (mxfp4, mxint4) or uint8 E4M3 (nvfp4); zeros: uint8
    [N, K/group] in [0, 15] for "uint4_zp", else None; global_scale: the per-tensor float32
    factor (NVFP4's second-level scale; 1 for the other formats).
    """
    if wfmt not in WFMTS:
        raise ValueError(wfmt)
    q = unpack_nibbles(codes)
    n, k = q.shape
    if k % group:
        raise ValueError("K must be a multiple of the group size")
    gidx = np.arange(k) // group                       # group of each K position
    s = scale_values(wfmt, scales)[:, gidx]            # [N, K]
    g = np.float64(np.float32(global_scale))
    if wfmt in ("int4_sym", "mxint4"):
        return F.int4_signed(q).astype(np.float64) * s * g
    if wfmt == "uint4_zp":
        z = np.asarray(zeros).astype(np.int64)[:, gidx]
        return (q.astype(np.int64) - z).astype(np.float64) * s * g
    return F.e2m1_to_float(q) * s * g


def dequant_bf16(wfmt, group, codes, scales, zeros=None):
    """The dequantized weights as BF16 numbers: RNE_bf16(W_exact), without the per-tensor
    scale (that one multiplies the output).  This is what a dequantization to BF16 must
    reproduce bit for bit; the GEMM's reference uses the exact weights."""
    return F.round_to_bf16(dequant(wfmt, group, codes, scales, zeros))


def gemm(x, w, chan_scale=None, tok_scale=None, bias=None):
    """y[m, n] = tok_scale[m] * chan_scale[n] * sum_k x[m, k] * w[n, k] + bias[n], in float64.

    x: activation values [M, K] (any real dtype, used exactly); w: exact weights [N, K].
    The bias is added after every scale ("Humming wird angekündigt", section "Gemeinsam
    genutzte CUDA-Komponenten": scaling and bias addition fused into the output stage).
    """
    y = np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T
    if tok_scale is not None:
        y = y * np.asarray(tok_scale, dtype=np.float64)[:, None]
    if chan_scale is not None:
        y = y * np.asarray(chan_scale, dtype=np.float64)[None, :]
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64)[None, :]
    return y


def w4a16(x_bits, wfmt, group, codes, scales, zeros=None, chan_scale=None, global_scale=1.0,
          bias=None):
    """Dense W4A16: BF16 activations (bit patterns [M, K]) times the exact dequantized weights.

    The plain definition: unpack the codes, dequantize exactly in float64 and multiply with
    float64 accumulation.  A kernel on a BF16 tensor core meets it by keeping the weights
    exact there and applying the group scale to its FP32 accumulators (the Chinese release
    notes, v0.1.3: the "apply scale on C" path); a BF16-rounded weight is what the
    dequantization check compares (dequant_bf16), not what the product uses.  The per-tensor
    scale (NVFP4) then multiplies the output like the per-channel one, and the bias b[n],
    if given, is added after every scale."""
    x = F.bf16_bits_to_float(x_bits)
    y = gemm(x, dequant(wfmt, group, codes, scales, zeros), chan_scale=chan_scale)
    y = y * np.float64(np.float32(global_scale))
    return y if bias is None else y + np.asarray(bias, dtype=np.float64)[None, :]


def quant_act_fp8(x_bits):
    """Tokenwise FP8 e4m3 activation quantization of BF16 rows.

    Returns (codes uint8 [M, K], scale float32 [M]).  Decisions are taken in float32: the
    row maximum, s = amax / 448, and the quotient x / s that is rounded to e4m3.
    """
    x = F.bf16_bits_to_float(x_bits).astype(np.float32)
    amax = np.max(np.abs(x), axis=1) if x.shape[1] else np.zeros(x.shape[0], np.float32)
    s = (amax.astype(np.float32) / np.float32(F.E4M3_MAX)).astype(np.float32)
    s = np.where(amax == 0, np.float32(1.0), s).astype(np.float32)
    v = (x / s[:, None]).astype(np.float32)            # IEEE float32 quotient
    return F.e4m3_encode(F.round_to_e4m3_satfinite(v.astype(np.float64))), s


def quant_act_mxfp4(x_bits, block=32):
    """MXFP4 activations: BF16 X [M, K] (bit patterns, K % block == 0) -> (codes uint8
    [M, K/2] in the canonical nibble order, E8M0 exponents uint8 [M, K/block])."""
    x = F.bf16_bits_to_float(x_bits)
    m, k = x.shape
    if k % block:
        raise ValueError("K must be a multiple of the block")
    xb = x.reshape(m, k // block, block)
    amax = np.max(np.abs(xb), axis=2)
    _, e2 = np.frexp(amax)                        # amax = f 2^e2 with 0.5 <= f < 1
    e = np.where(amax > 0, (e2 - 1) - 2 + 127, 127)   # floor(log2 amax) - 2, biased
    e = np.clip(e, 0, 254).astype(np.int64)
    q = F.round_to_e2m1_satfinite(xb / np.ldexp(1.0, e - 127)[..., None])
    nib = F.e2m1_encode(q).reshape(m, k)
    codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)   # even k in the low nibble
    return codes, e.astype(np.uint8)


def dequant_act_mxfp4(codes, exps, block=32):
    """The exact values of MXFP4 activations: e2m1(code) * 2^(E - 127) per block."""
    q = unpack_nibbles(codes)
    return F.e2m1_to_float(q) * F.e8m0_to_float(exps)[:, np.arange(q.shape[1]) // block]


def w4a4(xq, x_exps, wfmt, group, codes, scales, zeros=None, chan_scale=None, bias=None):
    """W4A4: y = sum_k dequant_act(xq)[m, k] * W[n, k] with exact weights (both operands are
    MX values a block-scaled FP4 MMA multiplies exactly), times c[n], plus b[n], if given."""
    return gemm(dequant_act_mxfp4(xq, x_exps), dequant(wfmt, group, codes, scales, zeros),
                chan_scale=chan_scale, bias=bias)


def w4a8(xq, tok_scale, wfmt, group, codes, scales, zeros=None, chan_scale=None, bias=None):
    """Dense W4A8: y = s_tok[m] * sum_k e4m3(xq[m, k]) * W[n, k]  (times c[n], plus b[n],
    if given)."""
    x = F.e4m3_to_float(xq)
    return gemm(x, dequant(wfmt, group, codes, scales, zeros),
                chan_scale=chan_scale, tok_scale=tok_scale, bias=bias)


def moe_grouped(x_rows, offsets, experts, tok_scale=None, chan_scales=None, biases=None):
    """MoE grouped GEMM over expert-sorted rows.

    x_rows: activation values [R, K] sorted by expert; offsets: int [E+1], rows
    offsets[e]..offsets[e+1] belong to expert e; experts: list of E exact weights [N, K].
    Each expert's block of rows is an ordinary dense GEMM with that expert's weights
    ("Humming wird angekündigt", section "WnA16": tokens are distributed over experts and
    the work per expert varies with the load).  biases: E bias vectors [N] or None, each
    added to its expert's rows after every scale.
    """
    x_rows = np.asarray(x_rows, dtype=np.float64)
    offsets = np.asarray(offsets, dtype=np.int64)
    n = experts[0].shape[0]
    y = np.zeros((x_rows.shape[0], n), dtype=np.float64)
    for e, w in enumerate(experts):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            ts = None if tok_scale is None else np.asarray(tok_scale)[a:b]
            cs = None if chan_scales is None else chan_scales[e]
            bs = None if biases is None else biases[e]
            y[a:b] = gemm(x_rows[a:b], w, chan_scale=cs, tok_scale=ts, bias=bs)
    return y


def moe_indexed(x, offsets, row_index, experts, tok_scale=None, biases=None):
    """MoE GEMM over rows gathered by index (the pages' "Indexed" MoE path, "Humming wird
    angekündigt", section "WnA16": the kernel reads each token's row where it lies instead
    of a copy sorted by expert).

    x: activation values [T, K] in token order; offsets: int [E+1] over the R sorted
    positions; row_index: int [R], the row of x that sorted position r takes, or a negative
    value for a padding position; experts: E exact weights [N, K]; tok_scale: float [T] per
    row of x (FP8 activations) or None; biases: E bias vectors [N] or None.  Output row r
    (sorted order) is x[row_index[r]] times expert e's weights for the e whose block holds
    r, scaled by tok_scale[row_index[r]], plus expert e's bias; padding positions give zero
    rows (the kernel's are unspecified).
    """
    x = np.asarray(x, dtype=np.float64)
    offsets = np.asarray(offsets, dtype=np.int64)
    row_index = np.asarray(row_index, dtype=np.int64)
    n = experts[0].shape[0]
    y = np.zeros((row_index.shape[0], n), dtype=np.float64)
    for e, w in enumerate(experts):
        for r in range(int(offsets[e]), int(offsets[e + 1])):
            t = int(row_index[r])
            if t < 0:
                continue
            ts = None if tok_scale is None else np.asarray(tok_scale)[t:t + 1]
            bs = None if biases is None else biases[e]
            y[r:r + 1] = gemm(x[t:t + 1], w, tok_scale=ts, bias=bs)
    return y


def tolerance_ok(y, y_ref, rel):
    """The parity bar: |y - y_ref| <= rel * max(|y_ref|, rms(y_ref)) elementwise.

    Returns (ok, worst ratio of error to the allowed bound)."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    if y_ref.size == 0:
        return True, 0.0
    rms = float(np.sqrt(np.mean(y_ref * y_ref)))
    bound = rel * np.maximum(np.abs(y_ref), rms)
    err = np.abs(y - y_ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / bound, np.where(err > 0, np.inf, 0.0))
    worst = float(np.max(ratio))
    return bool(worst <= 1.0 and np.all(np.isfinite(y))), worst
