"""W4A4: MXFP4 weights x MXFP4 activations on the block-scaled FP4 MMA ("Humming wird
angekündigt", section "W8A8 / W4A8 / W4A4": W4A4 with MX formats on Blackwell).

Checks: the activation quantization bit for bit against the oracle's OCP Microscaling
conversion; the W4A4 packed layout (codes in the MMA's own swizzled order) decoded back bit
for bit; an integer case where every partial sum is exact in FP32, so Y must be RNE_bf16 of
the oracle exactly; parity against the oracle (the exact MX values of both operands, float64
sum) for every token tile and schedule, with channel scale and bias; sampled parity at the
full MXFP4 shapes.  The bar is 2e-2 * max(|y_ref|, rms) like the other 8-bit-or-less
activation path, and every case logs its worst ratio."""
import numpy as np
import pytest
import torch

import oracle
from oracle import formats as F
import workloads as WL

pytestmark = pytest.mark.gpu

TOL_A4 = 2e-2


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


def _nan(M, N):
    return torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")


def _check(tag, y, ref):
    from tests import gpu_util as G
    G.log_parity(tag, y, ref, TOL_A4)
    ok, worst = oracle.tolerance_ok(y, ref, TOL_A4)
    assert ok, f"worst error / bound = {worst:.3f}"


def _quant(x_bits):
    from tests import gpu_util as G
    qg = _qg()
    Xq, E = qg.quant_act_mxfp4(G.bf16_tensor(x_bits))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    return Xq, E


@pytest.mark.parametrize("M,K", [(37, 544), (5, 7168), (64, 2048), (1, 32)])
def test_quant_act_mxfp4_bitexact(M, K):
    r = WL.rng(70)
    x = WL.gen_x(r, M, K, outliers=True)
    x[0, :32] = 0                                  # an all-zero block
    if K >= 64:
        x[0, 32:64] = WL.to_bf16_bits(np.full(32, 6.0, np.float32))   # amax exactly 6
    Xq, E = _quant(x)
    codes, exps = oracle.quant_act_mxfp4(x)
    np.testing.assert_array_equal(Xq.cpu().numpy(), codes)
    e = E.cpu().numpy()
    np.testing.assert_array_equal(e[:, :K // 32], exps)
    nb = (K // 32 + 3) // 4 * 4
    assert np.all(e[:, K // 32:nb] == 127)         # padding blocks of the last 128-K block


@pytest.mark.parametrize("N,K", [(300, 512), (128, 7168), (7168, 2048)])
def test_repack_w4a4_roundtrip(N, K):
    from tests import gpu_util as G
    qg = _qg()
    w = WL.gen_weights(WL.rng(71), "mxfp4", N, K)
    d, packed = G.pack(w, afmt="mxfp4")
    W = G.bf16_bits_of(qg.dequant_debug(d, packed))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    ref = F.float_to_bf16_bits(oracle.dequant_bf16(w.wfmt, w.group, w.codes, w.scales))
    both_zero = ((W & 0x7FFF) == 0) & ((ref & 0x7FFF) == 0)     # +0 and -0 are equal
    assert np.all((W == ref) | both_zero)


def _run(w, x, chan=None, bias=None, out=None):
    from tests import gpu_util as G
    qg = _qg()
    d, packed = G.pack(w, afmt="mxfp4")
    Xq, E = _quant(x)
    cs = None if chan is None else torch.from_numpy(chan).cuda()
    b = None if bias is None else torch.from_numpy(bias).cuda()
    y = qg.w4a4(d, packed, Xq, E, chan_scale=cs, bias=b, out=out if out is not None else _nan(x.shape[0], w.N))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    return G.to_f64(y), Xq.cpu().numpy(), E.cpu().numpy()


def test_w4a4_integer_inputs_exact():
    """X holds e2m1 grid values times 1 (block maxima 4 or 6 give E = 127), weight exponents
    in [124, 130]: every product is a multiple of 2^-5 and every partial sum stays below
    2^18, so the FP32 sums are exact and Y = RNE_bf16(oracle)."""
    r = WL.rng(72)
    M, N, K = 24, 256, 512
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -1.5, -2, -3, -4, -6], np.float32)
    xv = r.choice(grid, size=(M, K)).astype(np.float32)
    xv[:, ::32] = 6.0                               # every block's maximum is 6
    x = WL.to_bf16_bits(xv)
    w = WL.gen_weights(r, "mxfp4", N, K)
    w.scales[:] = r.integers(124, 131, size=w.scales.shape, dtype=np.uint8)
    y, xq, e = _run(w, x)
    ref = oracle.w4a4(xq, e[:, :K // 32], w.wfmt, w.group, w.codes, w.scales)
    np.testing.assert_array_equal(y, F.round_to_bf16(ref))


@pytest.mark.parametrize("tile", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("splits", [1, 3, -1])
def test_w4a4_every_tile(tile, splits):
    qg = _qg()
    r = WL.rng(73)
    M, N, K = 150, 384, 1024
    x = WL.gen_x(r, M, K, outliers=True)
    w = WL.gen_weights(r, "mxfp4", N, K)
    chan = r.uniform(0.5, 2.0, N).astype(np.float32)
    bias = r.standard_normal(N).astype(np.float32)
    qg.force_config(tile, splits)
    try:
        y, xq, e = _run(w, x, chan, bias)
    finally:
        qg.force_config(0, 0)
    ref = oracle.w4a4(xq, e[:, :K // 32], w.wfmt, w.group, w.codes, w.scales, chan_scale=chan,
                      bias=bias)
    _check(f"w4a4 tile {tile} splits {splits}", y, ref)


@pytest.mark.parametrize("M,N,K", [(1, 300, 544), (17, 129, 96), (300, 256, 2048)])
def test_w4a4_ragged(M, N, K):
    """N not a multiple of the 128-row tile, K not a multiple of the 128-K record (padded
    exponent words and zero codes past K), M across token tiles."""
    r = WL.rng(74)
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, "mxfp4", N, K)
    y, xq, e = _run(w, x)
    ref = oracle.w4a4(xq, e[:, :K // 32], w.wfmt, w.group, w.codes, w.scales)
    _check(f"w4a4 ragged {M}x{N}x{K}", y, ref)


@pytest.mark.parametrize("N,K,M", [(4096, 7168, 1), (7168, 2048, 16), (4096, 7168, 8192),
                                   (7168, 2048, 8192)])
def test_w4a4_bench_shapes(N, K, M):
    """The MXFP4 shapes of the bench, in the default plan: 64 weight rows x 48 token rows
    sampled against the oracle."""
    r = WL.rng(0)
    x = WL.gen_x(r, M, K, outliers=True)
    w = WL.gen_weights(r, "mxfp4", N, K)
    y, xq, e = _run(w, x)
    rs = WL.rng(75)
    ns = np.unique(np.concatenate([[0, N - 1], rs.choice(N, size=62, replace=False)]))
    ms = np.unique(np.concatenate([[0, M - 1], rs.choice(M, size=min(M, 46), replace=False)]))
    ref = oracle.w4a4(xq[ms], e[ms][:, :K // 32], w.wfmt, w.group, w.codes[ns], w.scales[ns])
    _check(f"fullsize w4a4 {N}x{K} M={M}", y[np.ix_(ms, ns)], ref)
