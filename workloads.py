"""Seeded synthetic inputs for the quantized-weight GEMM, shared by tests and the bench.

This module draws random numbers and lays them out in the library's canonical input
format; it contains none of the GEMM's arithmetic (no decoding, dequantization or
quantization).  Real numbers are drawn in float32 and rounded once to bfloat16 by
PyTorch's own conversion.  Every generator takes an explicit seed and draws its tensors
in a fixed order: X, codes, scales, zeros, then (MoE) router logits, outlier masks and the
second GEMM's input.

The workloads mirror the benchmark protocol of "Humming wird angekündigt" (vLLM blog,
German edition), section "Leistung": M over every power of two from 1 to 8192, each shape
timed alone with a cold L2; MoE speed-ups sum the gate_up and down GEMMs.  The shapes
named below stand in for the figures that the pages show but that did not survive.
"""
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

M_SWEEP = tuple(2 ** i for i in range(14))            # 1 .. 8192


@dataclass
class WeightCase:
    wfmt: str                  # "int4_sym" | "uint4_zp" | "mxfp4" | "mxint4" | "nvfp4"
    group: int
    N: int
    K: int
    codes: np.ndarray          # uint8 [N, K/2], even k in the low nibble
    scales: np.ndarray         # uint16 bf16 bits [N, K/g], uint8 E8M0 [N, K/32] or E4M3 [N, K/16]
    zeros: Optional[np.ndarray] = None   # uint8 [N, K/g] for uint4_zp
    global_scale: float = 1.0  # float32 per-tensor scale (nvfp4)


@dataclass
class MoECase:
    E: int
    topk: int
    T: int
    counts: np.ndarray         # int64 [E] routed (token, slot) pairs per expert, unpadded
    offsets: np.ndarray        # int32 [E+1] row offsets of each expert's padded block
    valid: np.ndarray          # bool [R] rows that carry a routed token (not padding)
    token_of_row: np.ndarray   # int64 [R] source token of each row (-1 for padding)
    x_bits: np.ndarray = field(default=None)        # uint16 [R, K] gate_up input, sorted
    down_bits: np.ndarray = field(default=None)     # uint16 [R, inter] down input
    x_tok_bits: np.ndarray = field(default=None)    # uint16 [T, K] gate_up input, token order


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16_bits(a):
    """float32 numpy array -> uint16 bf16 bit patterns (PyTorch's round-to-nearest-even)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def pack_nibbles(nib):
    """uint8 [N, K] values 0..15 -> uint8 [N, K/2] with even k in the low nibble."""
    nib = np.asarray(nib, dtype=np.uint8)
    return (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)


def gen_x(r, M, K, outliers=False):
    x = r.standard_normal((M, K), dtype=np.float32)
    if outliers:
        mask = r.random((M, K)) < 0.01
        x = np.where(mask, x * np.float32(20.0), x).astype(np.float32)
    return to_bf16_bits(x)


def gen_weights(r, wfmt, N, K, group=None, scale_lo=0.005, scale_hi=0.02, zp_lo=6, zp_hi=9,
                e8m0_lo=118, e8m0_hi=126, e4m3_exp_lo=5, e4m3_exp_hi=9, global_lo=0.002,
                global_hi=0.004):
    """Draw codes, then scales, then zero points or the per-tensor scale (in that order).

    mxfp4 / mxint4: all 16 codes, E8M0 exponents in [e8m0_lo, e8m0_hi] per 32.  nvfp4: all
    16 e2m1 codes, positive E4M3 scales with exponent field in [e4m3_exp_lo, e4m3_exp_hi]
    and any mantissa per 16, and a float32 per-tensor scale in [global_lo, global_hi)."""
    if wfmt in ("mxfp4", "mxint4"):
        group = 32 if group is None else group
        nib = r.integers(0, 16, size=(N, K), dtype=np.uint8)          # all 16 codes
        scales = r.integers(e8m0_lo, e8m0_hi + 1, size=(N, K // group), dtype=np.uint8)
        return WeightCase(wfmt, group, N, K, pack_nibbles(nib), scales)
    if wfmt == "nvfp4":
        group = 16 if group is None else group
        nib = r.integers(0, 16, size=(N, K), dtype=np.uint8)
        ex = r.integers(e4m3_exp_lo, e4m3_exp_hi + 1, size=(N, K // group))
        man = r.integers(0, 8, size=(N, K // group))
        scales = ((ex << 3) | man).astype(np.uint8)
        g = float(np.float32(r.uniform(global_lo, global_hi)))
        return WeightCase(wfmt, group, N, K, pack_nibbles(nib), scales, None, g)
    group = 128 if group is None else group
    if wfmt == "int4_sym":
        q = r.integers(-8, 8, size=(N, K), dtype=np.int64)             # signed codes
        nib = (q & 0xF).astype(np.uint8)                                # two's complement
    elif wfmt == "uint4_zp":
        nib = r.integers(0, 16, size=(N, K), dtype=np.uint8)
    else:
        raise ValueError(wfmt)
    s = r.uniform(scale_lo, scale_hi, size=(N, K // group)).astype(np.float32)
    scales = to_bf16_bits(s)
    zeros = None
    if wfmt == "uint4_zp":
        zeros = r.integers(zp_lo, zp_hi + 1, size=(N, K // group), dtype=np.uint8)
    return WeightCase(wfmt, group, N, K, pack_nibbles(nib), scales, zeros)


# ----------------------------------------------------------------------------------------
# The five seeded workloads.  Each function returns plain numpy arrays.

def tiny_dense(seed=0):
    """M=16, N=256, K=512, symmetric INT4, group 128, X ~ N(0,1)."""
    r = rng(seed)
    x = gen_x(r, 16, 512)
    w = gen_weights(r, "int4_sym", 256, 512, group=128)
    return x, w


def int4_asym_shape(N, K, M, seed=0):
    """Asymmetric INT4 (uint4 codes, zero points in [6, 9] per group of 128)."""
    r = rng(seed)
    x = gen_x(r, M, K)
    w = gen_weights(r, "uint4_zp", N, K, group=128)
    return x, w


def mxfp4_shape(N, K, M, seed=0, outliers=False):
    """MXFP4 weights (all 16 e2m1 codes, E8M0 exponents in [118, 126] per 32)."""
    r = rng(seed)
    x = gen_x(r, M, K, outliers=outliers)
    w = gen_weights(r, "mxfp4", N, K)
    return x, w


INT4_ASYM_SHAPES = ((28672, 8192), (8192, 28672))
MXFP4_SHAPES = ((4096, 7168), (7168, 2048))

MOE_E, MOE_TOPK, MOE_HIDDEN, MOE_INTER = 256, 8, 7168, 2048
MOE_T = (1, 16, 128, 1024, 8192)
MOE_PAD = 8


def route(r, T, E=MOE_E, topk=MOE_TOPK, skewed=False, pad=MOE_PAD):
    """Top-k routing over N(0,1) logits (+2 on experts 0..7 when skewed), then a stable
    sort of the (token, slot) pairs by expert and padding of each expert's block to a
    multiple of `pad` rows.  Softmax is monotonic, so the top-k of the softmax is the
    top-k of the logits; equal logits prefer the lower expert index."""
    logits = r.standard_normal((T, E), dtype=np.float32)
    if skewed:
        logits[:, :8] += np.float32(2.0)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :topk]        # [T, topk]
    pair_expert = order.reshape(-1)
    pair_token = np.repeat(np.arange(T), topk)
    sort = np.argsort(pair_expert, kind="stable")
    pair_expert, pair_token = pair_expert[sort], pair_token[sort]
    counts = np.bincount(pair_expert, minlength=E).astype(np.int64)
    padded = (counts + pad - 1) // pad * pad
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(padded)
    R = int(offsets[-1])
    token_of_row = np.full(R, -1, dtype=np.int64)
    start = 0
    for e in range(E):
        c = int(counts[e])
        token_of_row[offsets[e]:offsets[e] + c] = pair_token[start:start + c]
        start += c
    return counts, offsets.astype(np.int32), token_of_row >= 0, token_of_row


def moe_case(T, seed=0, skewed=False, E=MOE_E, topk=MOE_TOPK, hidden=MOE_HIDDEN,
             inter=MOE_INTER, with_inputs=True):
    """Routing plus the sorted gate_up input [R, hidden] and an independent down input
    [R, inter] (both bf16, padding rows zero).  Weights are drawn by moe_weights()."""
    r = rng(seed)
    x_tok = gen_x(r, T, hidden) if with_inputs else None
    counts, offsets, valid, tor = route(r, T, E, topk, skewed)
    case = MoECase(E, topk, T, counts, offsets, valid, tor)
    if with_inputs:
        R = len(tor)
        xs = np.zeros((R, hidden), dtype=np.uint16)
        xs[valid] = x_tok[tor[valid]]
        down = gen_x(r, R, inter)
        down[~valid] = 0
        case.x_bits, case.down_bits, case.x_tok_bits = xs, down, x_tok
    return case


def iter_moe_weights(E, N, K, seed=0):
    """The E experts' MXFP4 weights of one GEMM (gate_up: N=2*inter, K=hidden; down:
    N=hidden, K=inter), yielded expert by expert from one generator so that a caller can
    repack each and drop it.  Codes are drawn as whole bytes uniform over 0..255, which
    is two independent nibbles uniform over all 16 e2m1 codes; then the E8M0 exponents,
    uniform in [118, 126], one per 32 K-elements."""
    r = rng(seed + 1000)
    for _ in range(E):
        codes = np.frombuffer(bytearray(r.bytes(N * K // 2)), dtype=np.uint8).reshape(N, K // 2)
        scales = r.integers(118, 127, size=(N, K // 32), dtype=np.uint8)
        yield WeightCase("mxfp4", 32, N, K, codes, scales)


def moe_weights(E, N, K, seed=0):
    """All E experts of iter_moe_weights() as a list."""
    return list(iter_moe_weights(E, N, K, seed))
