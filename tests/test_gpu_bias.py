"""Fused bias in the output stage: y = (sum_k x w) * c[n] * s_tok[m] + b[n], one rounding to
BF16 ("Humming wird angekündigt", section "Gemeinsam genutzte CUDA-Komponenten": scaling and
bias addition fused into the output stage).  Parity against the float64 oracle for every
token tile and schedule (wide, narrow and cut-tile epilogues), the FP16-operand, BF16 and
NVFP4 output factors, FP8 activations with token scales, both MoE paths (a bias per expert)
and the host-buffer call."""
import numpy as np
import pytest
import torch

import oracle
from oracle import formats as F
import workloads as WL

pytestmark = pytest.mark.gpu

TOL_A16 = 8e-3
TOL_A8 = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    from quantized_weight_gemm_gb300 import build
    build.build()
    import quantized_weight_gemm_gb300 as qg
    qg.force_config(0, 0)
    qg.device_status(clear=True)
    yield
    qg.force_config(0, 0)
    assert qg.device_status(clear=True) == 0


def _qg():
    import quantized_weight_gemm_gb300 as qg
    return qg


def _f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _nan(M, N):
    return torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")


def _close(y, ref, tol):
    ok, worst = oracle.tolerance_ok(y, ref, tol)
    assert ok, f"worst error / bound = {worst:.3f}"


@pytest.mark.parametrize("wfmt", ["uint4_zp", "mxfp4", "nvfp4"])
@pytest.mark.parametrize("tile", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("splits", [1, 3, -1])
def test_bias_every_tile(wfmt, tile, splits):
    from tests import gpu_util as G
    qg = _qg()
    r = WL.rng(60)
    M, N, K = 150, 384, 1024
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, wfmt, N, K)
    chan = r.uniform(0.5, 2.0, N).astype(np.float32)
    bias = r.standard_normal(N).astype(np.float32)
    d, packed = G.pack(w)
    qg.force_config(tile, splits)
    try:
        y = qg.w4a16(d, packed, G.bf16_tensor(x), chan_scale=_f32(chan), bias=_f32(bias),
                     out=_nan(M, N))
        torch.cuda.synchronize()
    finally:
        qg.force_config(0, 0)
    assert qg.device_status(clear=True) == 0
    ref = oracle.w4a16(x, w.wfmt, w.group, w.codes, w.scales, w.zeros, chan_scale=chan,
                       global_scale=w.global_scale, bias=bias)
    _close(G.to_f64(y), ref, TOL_A16)


def test_bias_alone_is_exact():
    """Zero activations: Y is the bias rounded to BF16, bit for bit."""
    from tests import gpu_util as G
    qg = _qg()
    r = WL.rng(61)
    M, N, K = 40, 300, 512
    w = WL.gen_weights(r, "uint4_zp", N, K)
    bias = (r.standard_normal(N) * 3).astype(np.float32)
    d, packed = G.pack(w)
    X = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    y = G.to_f64(qg.w4a16(d, packed, X, bias=_f32(bias), out=_nan(M, N)))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    np.testing.assert_array_equal(y, np.broadcast_to(F.round_to_bf16(bias.astype(np.float64)), (M, N)))


@pytest.mark.parametrize("afmt", ["fp8", "fp8n"])
@pytest.mark.parametrize("tile,splits", [(16, 1), (32, -1), (64, 3), (128, 1), (256, 1)])
def test_bias_w4a8(tile, splits, afmt):
    """FP8 activations: token scale, channel scale and bias in one output expression."""
    from tests import gpu_util as G
    qg = _qg()
    r = WL.rng(62)
    M, N, K = 300, 256, 1024
    x = WL.gen_x(r, M, K, outliers=True)
    w = WL.gen_weights(r, "mxfp4", N, K)
    chan = r.uniform(0.5, 2.0, N).astype(np.float32)
    bias = r.standard_normal(N).astype(np.float32)
    d, packed = G.pack(w, afmt=afmt)
    xq, ts = oracle.quant_act_fp8(x)
    qg.force_config(tile, splits)
    try:
        y = qg.w4a8(d, packed, G.u8_tensor(xq), _f32(ts), chan_scale=_f32(chan), bias=_f32(bias),
                    out=_nan(M, N))
        torch.cuda.synchronize()
    finally:
        qg.force_config(0, 0)
    assert qg.device_status(clear=True) == 0
    ref = oracle.w4a8(xq, ts, w.wfmt, w.group, w.codes, w.scales, chan_scale=chan, bias=bias)
    _close(G.to_f64(y), ref, TOL_A8)


def _experts(r, wfmt, E, N, K):
    return [WL.gen_weights(r, wfmt, N, K) for _ in range(E)]


def _pack_experts(ws):
    from tests import gpu_util as G
    qg = _qg()
    d = G.desc_of(ws[0])
    codes = G.u8_tensor(np.stack([w.codes for w in ws]))
    sc = np.stack([w.scales for w in ws])
    sc = torch.from_numpy(sc.view(np.int16) if sc.dtype == np.uint16 else sc).cuda()
    z = None if ws[0].zeros is None else G.u8_tensor(np.stack([w.zeros for w in ws]))
    return d, qg.repack(d, codes, sc, z, num_experts=len(ws),
                        global_scale=[w.global_scale for w in ws])


def _exact(ws):
    return [oracle.dequant(w.wfmt, w.group, w.codes, w.scales, w.zeros) *
            np.float64(np.float32(w.global_scale)) for w in ws]


@pytest.mark.parametrize("wfmt", ["mxfp4", "uint4_zp"])
@pytest.mark.parametrize("stream_k", [False, True])
def test_bias_moe_grouped(wfmt, stream_k):
    from tests import gpu_util as G
    qg = _qg()
    r = WL.rng(63)
    N, K = 256, 1024
    counts = [5, 0, 37, 16, 0, 1, 130, 8]
    E = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    R = int(off[-1])
    x = WL.gen_x(r, R, K)
    ws = _experts(r, wfmt, E, N, K)
    biases = r.standard_normal((E, N)).astype(np.float32)
    d, packed = _pack_experts(ws)
    wsp = qg.moe_workspace(d, E, R) if stream_k else None
    y = qg.moe_grouped(d, packed, E, G.bf16_tensor(x), torch.tensor(off.astype(np.int32)).cuda(),
                       out=_nan(R, N), ws=wsp, bias=_f32(biases))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    ref = oracle.moe_grouped(F.bf16_bits_to_float(x), off, _exact(ws), biases=list(biases))
    _close(G.to_f64(y), ref, TOL_A16)


@pytest.mark.parametrize("wfmt", ["mxfp4", "uint4_zp"])
def test_bias_moe_indexed(wfmt):
    """Gathered rows (token order) with a bias per expert; padding positions are not
    compared (their outputs are unspecified)."""
    from tests import gpu_util as G
    qg = _qg()
    r = WL.rng(64)
    N, K, T, E = 256, 512, 40, 6
    counts = [7, 0, 12, 3, 25, 9]
    pad = [(c + 7) // 8 * 8 for c in counts]
    off = np.concatenate([[0], np.cumsum(pad)]).astype(np.int64)
    R = int(off[-1])
    idx = np.full(R, -1, dtype=np.int64)
    for e, c in enumerate(counts):
        idx[off[e]:off[e] + c] = r.integers(0, T, size=c)
    x = WL.gen_x(r, T, K)
    ws = _experts(r, wfmt, E, N, K)
    biases = r.standard_normal((E, N)).astype(np.float32)
    d, packed = _pack_experts(ws)
    y = qg.moe_indexed(d, packed, E, G.bf16_tensor(x), torch.tensor(off.astype(np.int32)).cuda(),
                       torch.tensor(idx.astype(np.int32)).cuda(), out=_nan(R, N),
                       bias=_f32(biases))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    ref = oracle.moe_indexed(F.bf16_bits_to_float(x), off, idx, _exact(ws), biases=list(biases))
    valid = idx >= 0
    _close(G.to_f64(y)[valid], ref[valid], TOL_A16)


def test_bias_host_buffers():
    """The host-buffer call forwards the bias to every chunk (3 chunks of 512 rows)."""
    from tests import gpu_util as G
    qg = _qg()
    r = WL.rng(65)
    M, N, K = 1300, 384, 512
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, "uint4_zp", N, K)
    bias = r.standard_normal(N).astype(np.float32)
    d, packed = G.pack(w)
    xh = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
    y = qg.w4a16_host(d, packed, xh, bias=_f32(bias))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    ref = oracle.w4a16(x, w.wfmt, w.group, w.codes, w.scales, w.zeros, bias=bias)
    _close(G.to_f64(y), ref, TOL_A16)
