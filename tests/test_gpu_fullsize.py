"""Parity at the full bench shapes, in the launch configuration the bench times (default plan):
sampled outputs checked against the float64 oracle one by one.

For each shape a GEMM runs over all N and M; 64 weight rows n (spread over the N tiles,
including the last) and up to 48 token rows m (including the first and last) are checked:
the oracle dequantizes only the sampled weight rows and multiplies them with the sampled
token rows.  The bar is the same element-wise tolerance as the small parity tests, with
rms(y_ref) taken over the sampled entries."""
import numpy as np
import pytest
import torch

import oracle
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
    assert qg.device_status(clear=True) == 0


def _samples(r, N, M):
    ns = np.unique(np.concatenate([[0, N - 1], r.choice(N, size=62, replace=False)]))
    ms = np.unique(np.concatenate([[0, M - 1], r.choice(M, size=min(M, 46), replace=False)]))
    return ns, ms


def _rows(w, ns):
    """The canonical tensors of the sampled weight rows only."""
    z = None if w.zeros is None else w.zeros[ns]
    return w.codes[ns], w.scales[ns], z


def _nan_out(M, N):
    """An output buffer whose every element the call must overwrite."""
    return torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")


@pytest.mark.parametrize("N,K,M", [(28672, 8192, 1), (28672, 8192, 16), (8192, 28672, 16),
                                   (28672, 8192, 256), (8192, 28672, 8192)])
def test_int4_zp_bench_shapes(N, K, M):
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    x, w = WL.int4_asym_shape(N, K, M, seed=0)
    d, packed = G.pack(w)
    y = qg.w4a16(d, packed, G.bf16_tensor(x), out=_nan_out(M, N))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    ns, ms = _samples(WL.rng(50), N, M)
    codes, scales, zeros = _rows(w, ns)
    ref = oracle.w4a16(x[ms], w.wfmt, w.group, codes, scales, zeros)
    got = y[torch.from_numpy(ms).cuda()][:, torch.from_numpy(ns).cuda()].double().cpu().numpy()
    ok, worst = oracle.tolerance_ok(got, ref, TOL_A16)
    assert ok, f"worst error / bound = {worst:.3f}"


@pytest.mark.parametrize("N,K,M", [(4096, 7168, 1), (7168, 2048, 16), (4096, 7168, 2048)])
def test_mxfp4_bench_shapes(N, K, M):
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    x, w = WL.mxfp4_shape(N, K, M, seed=0)
    d, packed = G.pack(w)
    y = qg.w4a16(d, packed, G.bf16_tensor(x), out=_nan_out(M, N))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    ns, ms = _samples(WL.rng(51), N, M)
    codes, scales, _ = _rows(w, ns)
    ref = oracle.w4a16(x[ms], w.wfmt, w.group, codes, scales)
    got = y[torch.from_numpy(ms).cuda()][:, torch.from_numpy(ns).cuda()].double().cpu().numpy()
    ok, worst = oracle.tolerance_ok(got, ref, TOL_A16)
    assert ok, f"worst error / bound = {worst:.3f}"


@pytest.mark.parametrize("N,K,M", [(4096, 7168, 1), (7168, 2048, 256), (4096, 7168, 8192)])
def test_w4a8_bench_shapes(N, K, M):
    """FP8 activations with 1% outliers, quantized by the library's own call; the oracle
    multiplies the same codes and scales (the quantization itself is checked bit for bit
    against the oracle in test_gpu_gemm)."""
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    x, w = WL.mxfp4_shape(N, K, M, seed=0, outliers=True)
    d, packed = G.pack(w, afmt="fp8")
    Xq, ts = qg.quant_act_fp8(G.bf16_tensor(x))
    y = qg.w4a8(d, packed, Xq, ts, out=_nan_out(M, N))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    ns, ms = _samples(WL.rng(52), N, M)
    codes, scales, _ = _rows(w, ns)
    mi = torch.from_numpy(ms).cuda()
    ref = oracle.w4a8(Xq[mi].cpu().numpy(), ts[mi].cpu().numpy(), w.wfmt, w.group, codes, scales)
    got = y[mi][:, torch.from_numpy(ns).cuda()].double().cpu().numpy()
    ok, worst = oracle.tolerance_ok(got, ref, TOL_A8)
    assert ok, f"worst error / bound = {worst:.3f}"
