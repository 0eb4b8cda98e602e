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


def _check_sampled(tag, y, x, w, ns, ms, tol=TOL_A16):
    """Sampled outputs against the exact weights; both worst ratios (exact, BF16-rounded
    weights) go to the parity log."""
    from tests import gpu_util as G
    codes, scales, zeros = _rows(w, ns)
    ref = oracle.w4a16(x[ms], w.wfmt, w.group, codes, scales, zeros, global_scale=w.global_scale)
    sub = WL.WeightCase(w.wfmt, w.group, len(ns), w.K, codes, scales, zeros, w.global_scale)
    got = y[torch.from_numpy(ms).cuda()][:, torch.from_numpy(ns).cuda()].double().cpu().numpy()
    G.log_parity(tag, got, ref, tol, G.ref_bf16_weights(x[ms], sub))
    ok, worst = oracle.tolerance_ok(got, ref, tol)
    assert ok, f"worst error / bound = {worst:.3f}"


@pytest.mark.parametrize("N,K,M", [(28672, 8192, 1), (28672, 8192, 16), (8192, 28672, 16),
                                   (8192, 28672, 1), (28672, 8192, 64), (8192, 28672, 128),
                                   (28672, 8192, 256), (28672, 8192, 1024),
                                   (8192, 28672, 2048), (8192, 28672, 8192),
                                   (28672, 8192, 8192)])
def test_int4_zp_bench_shapes(N, K, M):
    """Every token tile and schedule the INT4 sweep runs, including its dominant launch
    (N=28672, K=8192, M=8192)."""
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    x, w = WL.int4_asym_shape(N, K, M, seed=0)
    d, packed = G.pack(w)
    y = qg.w4a16(d, packed, G.bf16_tensor(x), out=_nan_out(M, N))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    ns, ms = _samples(WL.rng(50), N, M)
    _check_sampled(f"fullsize uint4_zp {N}x{K} M={M}", y, x, w, ns, ms)


def test_large_m_stream_k_gives_way_to_a_small_workspace():
    """Above M = 1024 with K >= 16384 the default plan runs stream-K over the leftover tiles;
    a workspace that holds only the activation copy gets whole tiles instead of an error.
    Both against the oracle on the same samples, and with each other."""
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    N, K, M = 8192, 28672, 1536
    x, w = WL.int4_asym_shape(N, K, M, seed=3)
    d, packed = G.pack(w)
    p = qg.plan(d, M)
    assert p["sk_tiles"] > 0 and p["max_contrib"] > 1
    X = G.bf16_tensor(x)
    ns, ms = _samples(WL.rng(52), N, M)
    y_sk = qg.w4a16(d, packed, X, out=_nan_out(M, N), ws=qg.workspace(d, M))
    small = torch.zeros(qg.act_copy_bytes(d, M), dtype=torch.uint8, device="cuda")
    y_whole = qg.w4a16(d, packed, X, out=_nan_out(M, N), ws=small)
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    _check_sampled(f"fullsize stream-K large M {N}x{K} M={M}", y_sk, x, w, ns, ms)
    _check_sampled(f"fullsize whole tiles large M {N}x{K} M={M}", y_whole, x, w, ns, ms)
    # the two schedules sum the same FP32 products in a different order
    diff = (y_sk.float() - y_whole.float()).abs().max().item()
    assert diff <= 8e-3 * y_whole.float().abs().max().item()


@pytest.mark.parametrize("N,K,M", [(4096, 7168, 1), (7168, 2048, 16), (4096, 7168, 2048),
                                   (7168, 2048, 1), (4096, 7168, 8192), (7168, 2048, 8192)])
def test_mxfp4_bench_shapes(N, K, M):
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    x, w = WL.mxfp4_shape(N, K, M, seed=0)
    d, packed = G.pack(w)
    y = qg.w4a16(d, packed, G.bf16_tensor(x), out=_nan_out(M, N))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    ns, ms = _samples(WL.rng(51), N, M)
    _check_sampled(f"fullsize mxfp4 {N}x{K} M={M}", y, x, w, ns, ms)


@pytest.mark.parametrize("wfmt", ["mxint4", "nvfp4"])
@pytest.mark.parametrize("N,K,M", [(4096, 7168, 1), (7168, 2048, 1), (4096, 7168, 8192),
                                   (7168, 2048, 8192)])
def test_mxint4_nvfp4_bench_shapes(wfmt, N, K, M):
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    r = WL.rng(0)
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, wfmt, N, K)
    d, packed = G.pack(w)
    y = qg.w4a16(d, packed, G.bf16_tensor(x), out=_nan_out(M, N))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    ns, ms = _samples(WL.rng(53), N, M)
    _check_sampled(f"fullsize {wfmt} {N}x{K} M={M}", y, x, w, ns, ms)


@pytest.mark.parametrize("afmt", ["fp8", "fp8n"])
@pytest.mark.parametrize("N,K,M", [(4096, 7168, 1), (7168, 2048, 256), (4096, 7168, 8192),
                                   (7168, 2048, 1), (7168, 2048, 8192)])
def test_w4a8_bench_shapes(N, K, M, afmt):
    """FP8 activations with 1% outliers, quantized by the library's own call; the oracle
    multiplies the same codes and scales (the quantization itself is checked bit for bit
    against the oracle in test_gpu_gemm)."""
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    x, w = WL.mxfp4_shape(N, K, M, seed=0, outliers=True)
    d, packed = G.pack(w, afmt=afmt)
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


@pytest.mark.parametrize("T", [1024, 8192])
@pytest.mark.parametrize("skewed", [False, True])
@pytest.mark.parametrize("gemm", ["gate_up", "down"])
def test_moe_layer_sampled(T, skewed, gemm):
    """Both grouped GEMMs of the 256-expert layer at prefill sizes, with the workspace the
    bench passes (stream-K over leftover tiles where the kernel takes it): 64 weight rows
    and 48 routed rows checked against the oracle, per expert of each sampled row."""
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    case = WL.moe_case(T, seed=0, skewed=skewed)
    N, K = (2 * WL.MOE_INTER, WL.MOE_HIDDEN) if gemm == "gate_up" else (WL.MOE_HIDDEN, WL.MOE_INTER)
    xb = case.x_bits if gemm == "gate_up" else case.down_bits
    E = case.E
    R = len(case.token_of_row)
    d = qg.WeightDesc("mxfp4", N, K, 32, "bf16")
    nb = qg.packed_bytes(d)
    packed = torch.empty(nb * E, dtype=torch.uint8, device="cuda")
    r = WL.rng(54)
    ns = np.unique(np.concatenate([[0, N - 1], r.choice(N, size=62, replace=False)]))
    valid_rows = np.nonzero(case.valid)[0]
    ms = np.unique(np.concatenate([valid_rows[[0, -1]], r.choice(valid_rows, size=46, replace=False)]))
    expert_of = np.searchsorted(case.offsets, ms, side="right") - 1
    need = set(int(e) for e in expert_of)
    rows_of = {}
    for e, w in enumerate(WL.iter_moe_weights(E, N, K, seed=0)):
        qg.repack(d, G.u8_tensor(w.codes), G.u8_tensor(w.scales), None,
                  out=packed[e * nb:(e + 1) * nb])
        if e in need:
            rows_of[e] = (w.codes[ns], w.scales[ns])
    X = G.bf16_tensor(xb)
    y = qg.moe_grouped(d, packed, E, X, torch.tensor(case.offsets, device="cuda"),
                       ws=qg.moe_workspace(d, E, R), out=_nan_out(R, N))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    ref = np.zeros((len(ms), len(ns)))
    for i, (m, e) in enumerate(zip(ms, expert_of)):
        codes, scales = rows_of[int(e)]
        ref[i] = oracle.w4a16(xb[[m]], "mxfp4", 32, codes, scales)[0]
    got = y[torch.from_numpy(ms).cuda()][:, torch.from_numpy(ns).cuda()].double().cpu().numpy()
    G.log_parity(f"fullsize moe {gemm} T={T} {'skewed' if skewed else 'uniform'}", got, ref, TOL_A16)
    ok, worst = oracle.tolerance_ok(got, ref, TOL_A16)
    assert ok, f"worst error / bound = {worst:.3f}"


@pytest.mark.parametrize("T", [16, 128])
@pytest.mark.parametrize("skewed", [False, True])
def test_moe_indexed_layer_matches_grouped(T, skewed):
    """The gate_up GEMM of the 256-expert layer at decode-to-prefill sizes on the indexed path
    with the bench's indexed workspace (from 256 sorted rows on: the rows gathered into it,
    then the grouped kernel; narrow tiles on FP16 operands): the same bits as the grouped
    call on the sorted rows, which matches the oracle on sampled rows."""
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    case = WL.moe_case(T, seed=1, skewed=skewed)
    N, K, E = 2 * WL.MOE_INTER, WL.MOE_HIDDEN, case.E
    R = len(case.token_of_row)
    assert R >= 256
    d = qg.WeightDesc("mxfp4", N, K, 32, "bf16")
    nb = qg.packed_bytes(d)
    packed = torch.empty(nb * E, dtype=torch.uint8, device="cuda")
    r = WL.rng(55)
    ns = np.unique(np.concatenate([[0, N - 1], r.choice(N, size=62, replace=False)]))
    valid_rows = np.nonzero(case.valid)[0]
    ms = np.unique(np.concatenate([valid_rows[[0, -1]],
                                   r.choice(valid_rows, size=min(46, len(valid_rows)), replace=False)]))
    expert_of = np.searchsorted(case.offsets, ms, side="right") - 1
    need = set(int(e) for e in expert_of)
    rows_of = {}
    for e, w in enumerate(WL.iter_moe_weights(E, N, K, seed=0)):
        qg.repack(d, G.u8_tensor(w.codes), G.u8_tensor(w.scales), None,
                  out=packed[e * nb:(e + 1) * nb])
        if e in need:
            rows_of[e] = (w.codes[ns], w.scales[ns])
    off = torch.tensor(case.offsets, device="cuda")
    y = qg.moe_grouped(d, packed, E, G.bf16_tensor(case.x_bits), off,
                       ws=qg.moe_workspace(d, E, R), out=_nan_out(R, N))
    idx = torch.from_numpy(case.token_of_row.astype(np.int32)).cuda()
    yi = qg.moe_indexed(d, packed, E, G.bf16_tensor(case.x_tok_bits), off, idx,
                        ws=qg.moe_indexed_workspace(d, E, T, R), out=_nan_out(R, N))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    assert torch.equal(y.view(torch.int16), yi.view(torch.int16))
    ref = np.zeros((len(ms), len(ns)))
    for i, (m, e) in enumerate(zip(ms, expert_of)):
        codes, scales = rows_of[int(e)]
        ref[i] = oracle.w4a16(case.x_bits[[m]], "mxfp4", 32, codes, scales)[0]
    got = yi[torch.from_numpy(ms).cuda()][:, torch.from_numpy(ns).cuda()].double().cpu().numpy()
    G.log_parity(f"fullsize moe indexed gate_up T={T} {'skewed' if skewed else 'uniform'}", got, ref,
                 TOL_A16)
    ok, worst = oracle.tolerance_ok(got, ref, TOL_A16)
    assert ok, f"worst error / bound = {worst:.3f}"


@pytest.mark.parametrize("wfmt", ["uint4_zp", "int4_sym", "mxint4"])
@pytest.mark.parametrize("tile", [32, 64, 128])
def test_cut_schedules_repeated(wfmt, tile):
    """Stream-K at the full 28672 x 8192 shape, called five times: a missing proxy fence
    between the dequant warps' reads of a record slot and its refill by bulk copy once
    decoded a lane quarter of a tile from the next record in most such calls."""
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    N, K, M = 28672, 8192, 64
    r = WL.rng(0)
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, wfmt, N, K)
    d, packed = G.pack(w)
    X = G.bf16_tensor(x)
    ns, ms = _samples(WL.rng(55), N, M)
    qg.force_config(tile, -1)
    try:
        for it in range(5):
            y = qg.w4a16(d, packed, X, out=_nan_out(M, N))
            torch.cuda.synchronize()
            assert qg.device_status(clear=True) == 0
            _check_sampled(f"fullsize stream-K {wfmt} tile {tile} call {it}", y, x, w, ns, ms)
    finally:
        qg.force_config(0, 0)
