"""Dense W4A16 / W4A8 parity of the CUDA path against the float64 oracle.

Bar: |y - y_ref| <= 8e-3 * max(|y_ref|, rms(y_ref)) for BF16 activations and 2e-2 for
FP8 activations, element by element; exact equality where the arithmetic is exact
(integer-valued inputs with power-of-two scales, one-hot activations)."""
import ctypes

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


def _run_a16(x_bits, w, chan=None):
    from tests import gpu_util as G
    qg = _qg()
    d, packed = G.pack(w)
    X = G.bf16_tensor(x_bits)
    cs = None if chan is None else torch.from_numpy(chan.astype(np.float32)).cuda()
    # NaN-filled output: an element the kernel does not write cannot pass for a result
    out = torch.full((X.shape[0], w.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = qg.w4a16(d, packed, X, chan_scale=cs, out=out)
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    return G.to_f64(y)


def _assert_close(y, ref, tol):
    ok, worst = oracle.tolerance_ok(y, ref, tol)
    if ok:
        return
    rms = np.sqrt(np.mean(ref * ref))
    ratio = np.abs(y - ref) / (tol * np.maximum(np.abs(ref), rms))
    bad = np.argwhere(~(ratio <= 1.0))
    m, n = (int(v) for v in np.unravel_index(np.nanargmax(np.where(np.isfinite(ratio), ratio, 1e30)), ratio.shape))
    rows = sorted(set(int(b[0]) for b in bad))
    cols = sorted(set(int(b[1]) for b in bad))
    raise AssertionError(
        f"worst error / bound = {worst:.3f} at (m={m}, n={n}): y={y[m, n]!r} ref={ref[m, n]!r}; "
        f"{len(bad)} of {ratio.size} bad; rows {rows[:12]}{'...' if len(rows) > 12 else ''} "
        f"({len(rows)}); cols {cols[:12]}{'...' if len(cols) > 12 else ''} ({len(cols)}); "
        f"bad n-tiles {sorted(set(c // 128 for c in cols))[:8]}")


def test_mxfp4_small_calls_fp16_operands():
    """MXFP4 weights with BF16 activations: a small call given a workspace runs on FP16
    operands (the hardware e2m1 conversion, the activations copied to FP16 by the
    pre-pass); with a workspace too small for that copy it runs on BF16 operands.  Both meet the bar against the exact
    weights.  Weight rows 0..127 have E8M0 exponents 165..200, rows 128..255 exponents
    100..110, more than 36 below the tensor's largest: on FP16 operands those blocks fall
    under FP16's subnormal grid (the rows' outputs become 0), far below the bar's
    max(|y|, rms(y)) scale, and the two paths differ exactly there."""
    from tests import gpu_util as G
    qg = _qg()
    r = WL.rng(38)
    M, N, K = 16, 256, 512
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, "mxfp4", N, K)
    w.scales[:128] = r.integers(165, 201, size=(128, K // 32), dtype=np.uint8)
    w.scales[128:] = r.integers(100, 111, size=(128, K // 32), dtype=np.uint8)
    d, packed = G.pack(w)
    X = G.bf16_tensor(x)
    qg.force_config(16, 1)                     # whole tiles: no workspace needed for cuts
    try:
        outs = {}
        # (a workspace too small for the activation copy keeps BF16 operands)
        small = torch.zeros(256, dtype=torch.uint8, device="cuda")
        for name, ws in (("f16", qg.workspace(d, M)), ("bf16", small)):
            out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            outs[name] = G.to_f64(qg.w4a16(d, packed, X, out=out, ws=ws))
            torch.cuda.synchronize()
            assert qg.device_status(clear=True) == 0
    finally:
        qg.force_config(0, 0)
    ref = oracle.w4a16(x, w.wfmt, w.group, w.codes, w.scales, w.zeros)
    for name in outs:
        _assert_close(outs[name], ref, TOL_A16)
    np.testing.assert_array_equal(outs["f16"][:, :128], outs["bf16"][:, :128])
    assert np.all(outs["f16"][:, 128:] == 0) and np.any(outs["bf16"][:, 128:] != 0)


def _check_a16(tag, y, x, w, chan=None):
    """The bar against the exact weights; both worst ratios (exact, BF16-rounded weights)
    go to the parity log."""
    from tests import gpu_util as G
    ref = oracle.w4a16(x, w.wfmt, w.group, w.codes, w.scales, w.zeros, chan_scale=chan,
                       global_scale=w.global_scale)
    G.log_parity(tag, y, ref, TOL_A16, G.ref_bf16_weights(x, w, chan))
    _assert_close(y, ref, TOL_A16)


def test_tiny_dense_workload():
    x, w = WL.tiny_dense(seed=0)
    _check_a16("tiny_dense", _run_a16(x, w), x, w)


@pytest.mark.parametrize("wfmt,group,M,N,K", [
    ("uint4_zp", 128, 37, 300, 1024),
    ("uint4_zp", 128, 1, 512, 2048),
    ("int4_sym", 128, 129, 256, 512),
    ("int4_sym", 32, 200, 129, 96),
    ("uint4_zp", 64, 300, 640, 512),
    ("uint4_zp", 256, 65, 384, 768),
    ("mxfp4", 32, 5, 520, 2048),
    ("mxfp4", 32, 17, 1024, 1024),
    ("mxfp4", 32, 260, 256, 416),
    ("mxfp4", 32, 600, 384, 640),
    ("mxint4", 32, 5, 520, 2048),
    ("mxint4", 32, 260, 256, 416),
    ("nvfp4", 16, 1, 512, 7168),
    ("nvfp4", 16, 17, 1024, 1024),
    ("nvfp4", 16, 600, 384, 640),
])
def test_dense_a16_parity(wfmt, group, M, N, K):
    r = WL.rng(21)
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, wfmt, N, K, group=group)
    _check_a16(f"dense_a16 {wfmt} g{group} {M}x{N}x{K}", _run_a16(x, w), x, w)


def test_chan_scale():
    r = WL.rng(22)
    x = WL.gen_x(r, 48, 512)
    w = WL.gen_weights(r, "uint4_zp", 200, 512)
    chan = r.uniform(0.5, 2.0, 200).astype(np.float32)
    _check_a16("chan_scale uint4_zp", _run_a16(x, w, chan), x, w, chan)


def test_nvfp4_chan_and_global_scale():
    """The per-channel and the per-tensor scale multiply the same output."""
    r = WL.rng(25)
    x = WL.gen_x(r, 48, 512)
    w = WL.gen_weights(r, "nvfp4", 200, 512)
    chan = r.uniform(0.5, 2.0, 200).astype(np.float32)
    ref = oracle.w4a16(x, w.wfmt, w.group, w.codes, w.scales, chan_scale=chan,
                       global_scale=w.global_scale)
    _assert_close(_run_a16(x, w, chan), ref, TOL_A16)


@pytest.mark.parametrize("wfmt,group", [("int4_sym", 128), ("uint4_zp", 64), ("mxfp4", 32),
                                        ("mxint4", 32), ("nvfp4", 16)])
def test_integer_inputs_exact(wfmt, group):
    """Integer X and power-of-two scales: every partial sum is exact in fp32, so the
    output must be exactly RNE_bf16 of the oracle's exact result."""
    r = WL.rng(23)
    M, N, K = 8, 256, 256
    x = WL.to_bf16_bits(r.integers(-4, 5, size=(M, K)).astype(np.float32))
    w = WL.gen_weights(r, wfmt, N, K, group=group)
    if wfmt in ("mxfp4", "mxint4"):
        w.scales[:] = r.integers(124, 130, size=w.scales.shape, dtype=np.uint8)
    elif wfmt == "nvfp4":
        w.scales[:] = (r.integers(4, 10, size=w.scales.shape) << 3).astype(np.uint8)  # 2^-3..2^2
        w.global_scale = 0.25
    else:
        w.scales[:] = F.float_to_bf16_bits(np.ldexp(1.0, r.integers(-3, 3, size=w.scales.shape)))
    ref = oracle.w4a16(x, w.wfmt, w.group, w.codes, w.scales, w.zeros,
                       global_scale=w.global_scale)
    y = _run_a16(x, w)
    np.testing.assert_array_equal(y, F.round_to_bf16(ref))


@pytest.mark.parametrize("wfmt,group", [("uint4_zp", 128), ("mxfp4", 32), ("mxint4", 32),
                                        ("nvfp4", 16)])
def test_one_hot_columns_exact(wfmt, group):
    r = WL.rng(24)
    N, K = 384, 512
    w = WL.gen_weights(r, wfmt, N, K, group=group)
    w.global_scale = 0.125 if wfmt == "nvfp4" else 1.0      # a power of two: one rounding
    ks = np.array([0, 1, 31, 32, 63, 64, 127, 128, 255, 511])
    x = np.zeros((len(ks), K), dtype=np.float32)
    x[np.arange(len(ks)), ks] = 1.0
    y = _run_a16(WL.to_bf16_bits(x), w)
    W = oracle.dequant(w.wfmt, w.group, w.codes, w.scales, w.zeros, w.global_scale)
    if wfmt in ("int4_sym", "uint4_zp"):
        # INT4 with BF16 scales runs on FP16 operands: the weight reaches the tensor core
        # rounded to FP16's 11 significant bits (times a power of two), then Y is rounded
        # to BF16
        m, e = np.frexp(W)
        W = np.ldexp(np.rint(m * 2.0 ** 11) / 2.0 ** 11, e)
    np.testing.assert_array_equal(y, F.round_to_bf16(W)[:, ks].T)


@pytest.mark.parametrize("wfmt", ["mxint4", "nvfp4"])
@pytest.mark.parametrize("tile", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("splits", [1, 3, -1])
def test_new_formats_every_tile(wfmt, tile, splits):
    """Each token tile (wide, narrow and cut-tile epilogues) and K cut, for the formats whose
    decode (and, for NVFP4, output factor) the kernels compile separately."""
    qg = _qg()
    r = WL.rng(26)
    M, N, K = 150, 384, 1024
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, wfmt, N, K)
    ref = oracle.w4a16(x, w.wfmt, w.group, w.codes, w.scales, global_scale=w.global_scale)
    qg.force_config(tile, splits)
    try:
        y = _run_a16(x, w)
    finally:
        qg.force_config(0, 0)
    _assert_close(y, ref, TOL_A16)


@pytest.mark.parametrize("wfmt,afmt", [("uint4_zp", "bf16"), ("mxfp4", "bf16"),
                                       ("nvfp4", "bf16"), ("mxfp4", "fp8"), ("mxfp4", "fp8n")])
def test_batch_invariant_rows(wfmt, afmt):
    """With the batch-invariant flag, row m of Y is the same bits for every M (the default
    schedules change token tile and K cuts with M), and the largest call matches the oracle."""
    from tests import gpu_util as G
    qg = _qg()
    r = WL.rng(27)
    Mmax, N, K = 1000, 384, 1536
    x = WL.gen_x(r, Mmax, K, outliers=(afmt != "bf16"))
    w = WL.gen_weights(r, wfmt, N, K)
    d = qg.WeightDesc(wfmt, N, K, w.group, afmt, batch_invariant=True)
    z = None if w.zeros is None else G.u8_tensor(w.zeros)
    packed = qg.repack(d, G.u8_tensor(w.codes), G.scales_tensor(w), z, global_scale=w.global_scale)
    X = G.bf16_tensor(x)
    if afmt != "bf16":
        Xq, ts = qg.quant_act_fp8(X)
        run = lambda M: qg.w4a8(d, packed, Xq[:M], ts[:M])
    else:
        run = lambda M: qg.w4a16(d, packed, X[:M])
    full = G.bf16_bits_of(run(Mmax))
    for M in (1, 5, 64, 129, 700):
        np.testing.assert_array_equal(G.bf16_bits_of(run(M)), full[:M])
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    y = F.bf16_bits_to_float(full)
    if afmt != "bf16":
        xq, s = oracle.quant_act_fp8(x)
        ref = oracle.w4a8(xq, s, w.wfmt, w.group, w.codes, w.scales)
        _assert_close(y, ref, TOL_A8)
    else:
        ref = oracle.w4a16(x, w.wfmt, w.group, w.codes, w.scales, w.zeros,
                           global_scale=w.global_scale)
        _assert_close(y, ref, TOL_A16)


def test_batch_invariant_host_chunks():
    """The host-buffer call cuts M into chunks; with the flag every chunk's rows are the same
    bits as the device call on all rows."""
    from tests import gpu_util as G
    qg = _qg()
    r = WL.rng(28)
    M, N, K = 1500, 256, 1024
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, "uint4_zp", N, K)
    d = qg.WeightDesc("uint4_zp", N, K, 128, batch_invariant=True)
    packed = qg.repack(d, G.u8_tensor(w.codes), G.scales_tensor(w), G.u8_tensor(w.zeros))
    X = G.bf16_tensor(x)
    dev = G.bf16_bits_of(qg.w4a16(d, packed, X))
    xh = X.cpu().pin_memory()
    yh = qg.w4a16_host(d, packed, xh)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(yh.view(torch.int16).numpy().view(np.uint16), dev)


@pytest.mark.parametrize("N,K,M", [(19968, 512, 16), (6400, 256, 16), (19968, 512, 1)])
def test_default_plan_small_k(N, K, M):
    """Small-K shapes with the planner's own choice.  On 152 SMs, 19968 x 512 at M = 16 is
    one whole round of tiles plus four leftover tiles of four records each, cut over
    stream-K with fewer records than CTAs."""
    qg = _qg()
    r = WL.rng(29)
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, "uint4_zp", N, K)
    ref = oracle.w4a16(x, w.wfmt, w.group, w.codes, w.scales, w.zeros)
    _assert_close(_run_a16(x, w), ref, TOL_A16)


@pytest.mark.parametrize("tile", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("splits", [1, 2, 3, 7, -1])
def test_every_dispatch_entry(tile, splits):
    """Each (token tile, schedule) configuration the dispatcher can pick, forced: uniform K
    cuts and stream-K (-1; here every tile is shared by up to eight CTAs)."""
    qg = _qg()
    r = WL.rng(25)
    M, N, K = 100, 384, 1024
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, "uint4_zp", N, K)
    ref = oracle.w4a16(x, w.wfmt, w.group, w.codes, w.scales, w.zeros)
    qg.force_config(tile, splits)
    try:
        y = _run_a16(x, w)
        y2 = _run_a16(x, w)            # the workspace must come back zeroed
    finally:
        qg.force_config(0, 0)
    _assert_close(y, ref, TOL_A16)
    _assert_close(y2, ref, TOL_A16)


# ------------------------------------------------------------------------------- W4A8

@pytest.mark.parametrize("M,splits", [(16, 2), (16, 3), (16, 5), (16, -1), (100, -1)])
def test_many_units_with_odd_stage_counts(M, splits):
    """Many units per CTA whose stage counts are odd or differ between units: the stage
    to warp assignment runs on across unit boundaries and must keep every ring slot with
    fixed owners (a slot shared by two waiters lets one of them pass a wait a phase early).
    Stream-K (-1) here cuts the 72 (M = 16) or 48 (M = 100, seven token tiles) leftover
    tiles into pieces of a few K blocks, then runs whole tiles."""
    qg = _qg()
    r = WL.rng(30)
    N, K = 28672, 1152                                # 224 weight tiles x 9 K-blocks
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, "uint4_zp", N, K)
    ref = oracle.w4a16(x, w.wfmt, w.group, w.codes, w.scales, w.zeros)
    qg.force_config(16, splits)
    try:
        y = _run_a16(x, w)
    finally:
        qg.force_config(0, 0)
    _assert_close(y, ref, TOL_A16)


@pytest.mark.parametrize("M,K", [(67, 1000), (3, 1001), (5, 28672), (2, 7168), (9, 24)])
def test_quant_act_fp8_bitexact(M, K):
    """Vector path (K % 8 == 0; rows longer than the register-kept part re-read) and the
    scalar path (K = 1001)."""
    from tests import gpu_util as G
    qg = _qg()
    r = WL.rng(26)
    x = WL.gen_x(r, M, K, outliers=True)
    x[min(1, M - 1)] = 0                             # an all-zero row
    codes, s = qg.quant_act_fp8(G.bf16_tensor(x))
    ref_codes, ref_s = oracle.quant_act_fp8(x)
    np.testing.assert_array_equal(s.cpu().numpy(), ref_s)
    np.testing.assert_array_equal(codes.cpu().numpy(), ref_codes)


# The two W4A8 kernels: e2m1 -> e4m3 in registers ("fp8"), and the e2m1 codes as FP4
# tensor-core operands ("fp8n").
A8_FORMS = ["fp8", "fp8n"]


def _run_a8(xq, s, w, chan=None, afmt="fp8"):
    from tests import gpu_util as G
    qg = _qg()
    d, packed = G.pack(w, afmt=afmt)
    cs = None if chan is None else torch.from_numpy(chan.astype(np.float32)).cuda()
    out = torch.full((xq.shape[0], w.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = qg.w4a8(d, packed, G.u8_tensor(xq), torch.from_numpy(s).cuda(), chan_scale=cs, out=out)
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    return G.to_f64(y)


@pytest.mark.parametrize("afmt", A8_FORMS)
@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (16, 300, 1024), (40, 512, 2048),
                                   (130, 256, 384), (300, 640, 1024)])
def test_dense_a8_parity(M, N, K, afmt):
    r = WL.rng(27)
    x = WL.gen_x(r, M, K, outliers=True)
    w = WL.gen_weights(r, "mxfp4", N, K)
    xq, s = oracle.quant_act_fp8(x)
    ref = oracle.w4a8(xq, s, w.wfmt, w.group, w.codes, w.scales)
    _assert_close(_run_a8(xq, s, w, afmt=afmt), ref, TOL_A8)


@pytest.mark.parametrize("afmt", A8_FORMS)
def test_a8_integer_inputs_exact(afmt):
    r = WL.rng(28)
    M, N, K = 8, 256, 256
    xq = F.e4m3_encode(r.integers(-4, 5, size=(M, K)).astype(np.float64))
    s = np.ones(M, dtype=np.float32)
    w = WL.gen_weights(r, "mxfp4", N, K)
    w.scales[:] = r.integers(124, 130, size=w.scales.shape, dtype=np.uint8)
    ref = oracle.w4a8(xq, s, w.wfmt, w.group, w.codes, w.scales)
    np.testing.assert_array_equal(_run_a8(xq, s, w, afmt=afmt), F.round_to_bf16(ref))


@pytest.mark.parametrize("afmt", A8_FORMS)
@pytest.mark.parametrize("tile", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("splits", [1, 3, -1])
def test_a8_dispatch_entries(tile, splits, afmt):
    qg = _qg()
    r = WL.rng(29)
    M, N, K = 100, 384, 1024
    x = WL.gen_x(r, M, K, outliers=True)
    w = WL.gen_weights(r, "mxfp4", N, K)
    xq, s = oracle.quant_act_fp8(x)
    chan = r.uniform(0.5, 2, N).astype(np.float32)
    ref = oracle.w4a8(xq, s, w.wfmt, w.group, w.codes, w.scales, chan_scale=chan)
    qg.force_config(tile, splits)
    try:
        y = _run_a8(xq, s, w, chan, afmt=afmt)
    finally:
        qg.force_config(0, 0)
    _assert_close(y, ref, TOL_A8)


# ------------------------------------------------------------------- host buffers

@pytest.mark.parametrize("M,ldx_pad,ldy_pad", [(1, 0, 0), (300, 0, 0), (1500, 8, 16),
                                               (2049, 0, 8), (5000, 0, 0)])
def test_w4a16_host_buffers(M, ldx_pad, ldy_pad):
    """X and Y in page-locked host memory: one chunk (M <= 512) or several (chunks of at
    least 512 rows, the last one ragged: 1500 = 2 x 512 + 476, 5000 = 9 x 512 + 392), leading dimensions wider than K and N;
    the padding columns of Y stay untouched, and a second call on the same staging buffer
    gives the same bits."""
    from tests import gpu_util as G
    qg = _qg()
    r = WL.rng(34)
    N, K = 1024, 512
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, "uint4_zp", N, K)
    ref = oracle.w4a16(x, w.wfmt, w.group, w.codes, w.scales, w.zeros)
    d, packed = G.pack(w)
    xh = torch.zeros(M, K + ldx_pad, dtype=torch.bfloat16).pin_memory()
    xh[:, :K] = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    yh = torch.full((M, N + ldy_pad), 7.0, dtype=torch.bfloat16).pin_memory()
    staging = qg.host_staging(d, M)
    ws = qg.workspace(d, M)
    qg.w4a16_host(d, packed, xh[:, :K], out=yh[:, :N], staging=staging, ws=ws)
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    y1 = yh[:, :N].float().numpy().astype(np.float64)
    _assert_close(y1, ref, TOL_A16)
    if ldy_pad:
        assert torch.all(yh[:, N:] == 7.0)
    qg.w4a16_host(d, packed, xh[:, :K], out=yh[:, :N], staging=staging, ws=ws)
    torch.cuda.synchronize()
    assert np.array_equal(yh[:, :N].float().numpy().astype(np.float64), y1)


def test_w4a16_host_argument_errors():
    from tests import gpu_util as G
    qg = _qg()
    w = WL.gen_weights(WL.rng(35), "int4_sym", 256, 512)
    d, packed = G.pack(w)
    L = qg.lib()
    cd = d.c()
    P = ctypes.c_void_p
    xh = torch.zeros(600, 512, dtype=torch.bfloat16).pin_memory()
    yh = torch.zeros(600, 256, dtype=torch.bfloat16).pin_memory()
    need = qg.host_staging_bytes(d, 600)
    assert need == 2 * (512 * 512 * 2 + 256 * 512 * 2)          # chunks of 512 rows
    st = torch.empty(need, dtype=torch.uint8, device="cuda")
    args = lambda stg, n: (ctypes.byref(cd), P(packed.data_ptr()), P(xh.data_ptr()), 600, 512, None,
                           None, P(yh.data_ptr()), 256, stg, n, None, 0, None)
    assert L.qgemm_w4a16_host(*args(None, 0)) == 4                    # no staging
    assert L.qgemm_w4a16_host(*args(P(st.data_ptr()), need - 1)) == 4  # too small
    assert L.qgemm_w4a16_host(*args(P(st.data_ptr() + 16), need)) == 3  # misaligned
    assert L.qgemm_w4a16_host(ctypes.byref(cd), P(packed.data_ptr()), None, 600, 512, None, None,
                              P(yh.data_ptr()), 256, P(st.data_ptr()), need, None, 0, None) == 1


def test_w4a16_host_channel_scale():
    """The host-buffer call forwards the per-channel scale to every chunk (3 chunks)."""
    from tests import gpu_util as G
    qg = _qg()
    r = WL.rng(36)
    M, N, K = 1300, 768, 640
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, "mxfp4", N, K)
    chan = r.uniform(0.25, 4.0, size=N).astype(np.float32)
    ref = oracle.w4a16(x, w.wfmt, w.group, w.codes, w.scales, w.zeros, chan_scale=chan)
    d, packed = G.pack(w)
    xh = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
    y = qg.w4a16_host(d, packed, xh, chan_scale=torch.from_numpy(chan).cuda())
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    _assert_close(y.float().numpy().astype(np.float64), ref, TOL_A16)
