"""MoE grouped GEMM parity of the CUDA path against the float64 oracle.

Rows X_sorted[offsets[e]:offsets[e+1]] are multiplied by expert e's weights ("Humming wird
angekündigt", section "WnA16": tokens are distributed over the experts and the work per
expert varies with the load).  Covered: empty experts, counts that are not a multiple of
the token tile, the padded blocks the router produces, E = 1 reducing to the dense call,
both activation formats, every token tile, and sampled rows of the DeepSeek-V3-like layer
(E = 256, top-8, hidden 7168, expert intermediate 2048)."""
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
    qg.force_config(0, 0)
    assert qg.device_status(clear=True) == 0


def _stack(ws, field):
    a = [getattr(w, field) for w in ws]
    if a[0] is None:
        return None
    return np.stack(a)


def _pack_experts(ws, afmt="bf16"):
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    d = G.desc_of(ws[0], afmt)
    codes = G.u8_tensor(_stack(ws, "codes"))
    sc = _stack(ws, "scales")
    sc = torch.from_numpy(sc.view(np.int16) if sc.dtype == np.uint16 else sc).cuda()
    z = _stack(ws, "zeros")
    z = None if z is None else G.u8_tensor(z)
    return d, qg.repack(d, codes, sc, z, num_experts=len(ws),
                        global_scale=[w.global_scale for w in ws])


def _experts_a16(ws):
    """The exact weights times each expert's per-tensor scale (which multiplies its output,
    so it may as well scale its weights: the oracle sums exactly)."""
    return [oracle.dequant(w.wfmt, w.group, w.codes, w.scales, w.zeros) *
            np.float64(np.float32(w.global_scale)) for w in ws]


def _experts_exact(ws):
    return [oracle.dequant(w.wfmt, w.group, w.codes, w.scales, w.zeros) for w in ws]


def _run_moe(ws, x_bits, offsets, afmt="bf16", tok_scale=None, out_fill=float("nan"),
             stream_k=False, calls=1):
    """stream_k: pass the MoE workspace, which lets the kernel cut leftover tiles over CTAs
    (it does so when the leftover tiles hold at least 16 K blocks per SM)."""
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    d, packed = _pack_experts(ws, afmt)
    off = torch.tensor(np.asarray(offsets, dtype=np.int32), device="cuda")
    R = x_bits.shape[0]
    wsp = qg.moe_workspace(d, len(ws), R) if stream_k else None
    out = torch.empty(R, ws[0].N, dtype=torch.bfloat16, device="cuda")
    for _ in range(calls):            # later calls check that the workspace came back clean
        if out_fill is not None:
            out.fill_(out_fill)
        if afmt == "bf16":
            X = G.bf16_tensor(x_bits)
            y = qg.moe_grouped(d, packed, len(ws), X, off, out=out, ws=wsp)
        else:
            X = G.u8_tensor(x_bits)
            ts = torch.from_numpy(np.asarray(tok_scale, dtype=np.float32)).cuda()
            y = qg.moe_grouped(d, packed, len(ws), X, off, tok_scale=ts, out=out, ws=wsp)
        torch.cuda.synchronize()
        assert qg.device_status(clear=True) == 0
    return G.to_f64(y)


def _assert_close(y, ref, tol, rows=None):
    if rows is not None:
        y, ref = y[rows], ref[rows]
    ok, worst = oracle.tolerance_ok(y, ref, tol)
    assert ok, f"worst error / bound = {worst:.3f}"


def _offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)


@pytest.mark.parametrize("stream_k", [False, True])
@pytest.mark.parametrize("wfmt,counts,N,K", [
    ("mxfp4", [5, 0, 37, 16, 0, 1, 130, 8], 256, 512),
    ("mxfp4", [0, 0, 0, 64], 384, 1024),
    ("uint4_zp", [17, 300, 0, 3], 300, 768),
    ("int4_sym", [1, 1, 1, 1, 1, 1, 1, 1, 1, 1], 128, 256),
    ("mxint4", [9, 0, 70, 2], 256, 512),
    ("nvfp4", [5, 0, 37, 16, 0, 1, 130, 8], 256, 512),
])
def test_moe_a16_parity(wfmt, counts, N, K, stream_k):
    r = WL.rng(41)
    off = _offsets(counts)
    R = int(off[-1])
    x = WL.gen_x(r, R, K)
    ws = [WL.gen_weights(r, wfmt, N, K) for _ in counts]
    ref = oracle.moe_grouped(F_bits(x), off, _experts_a16(ws))
    _assert_close(_run_moe(ws, x, off, stream_k=stream_k, calls=2), ref, TOL_A16)


def F_bits(x_bits):
    from oracle import formats as F
    return F.bf16_bits_to_float(x_bits)


@pytest.mark.parametrize("afmt,counts,N,K", [
    ("bf16", [1, 1, 2, 1, 1, 1, 1, 1], 7168, 3072),     # 448 tiles: two whole rounds, 144 cut
    ("bf16", [1, 1, 1, 1, 1, 1, 1, 1], 2048, 2560),     # 128 tiles, all cut (20 K blocks each)
    ("bf16", [40, 3, 0, 17, 9, 1, 0, 22], 1536, 2688),  # several m-tiles per expert
    ("fp8", [12, 0, 41, 200, 1], 2048, 3584),           # 64-row tiles, FP8 activations
    ("fp8n", [12, 0, 41, 200, 1], 2048, 3584),          # ... on FP4 tensor-core operands
])
def test_moe_stream_k(afmt, counts, N, K):
    """MoE calls whose leftover tiles hold at least 16 K blocks per SM, so that the kernel
    cuts them over several CTAs (given the workspace); two calls on one workspace."""
    r = WL.rng(46)
    off = _offsets(counts)
    R = int(off[-1])
    x = WL.gen_x(r, R, K, outliers=afmt != "bf16")
    ws = [WL.gen_weights(r, "mxfp4", N, K) for _ in counts]
    if afmt == "bf16":
        ref = oracle.moe_grouped(F_bits(x), off, _experts_a16(ws))
        _assert_close(_run_moe(ws, x, off, stream_k=True, calls=2), ref, TOL_A16)
    else:
        from oracle import formats as F
        xq, sc = oracle.quant_act_fp8(x)
        ref = oracle.moe_grouped(F.e4m3_to_float(xq), off, _experts_exact(ws), tok_scale=sc)
        _assert_close(_run_moe(ws, xq, off, afmt=afmt, tok_scale=sc, stream_k=True, calls=2),
                      ref, TOL_A8)


@pytest.mark.parametrize("tile", [16, 32, 64, 128, 256])
def test_moe_every_token_tile(tile):
    import quantized_weight_gemm_gb300 as qg
    r = WL.rng(42)
    counts = [3, 70, 0, 129, 16, 33]
    off = _offsets(counts)
    R = int(off[-1])
    N, K = 256, 640
    x = WL.gen_x(r, R, K)
    ws = [WL.gen_weights(r, "mxfp4", N, K) for _ in counts]
    ref = oracle.moe_grouped(F_bits(x), off, _experts_a16(ws))
    qg.force_config(tile, 0)
    try:
        y = _run_moe(ws, x, off)
        y2 = _run_moe(ws, x, off, stream_k=True)
    finally:
        qg.force_config(0, 0)
    _assert_close(y, ref, TOL_A16)
    _assert_close(y2, ref, TOL_A16)


def test_moe_single_expert_equals_dense():
    """E = 1 over all rows is the dense call (same kernel schedule reduced to one group)."""
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    r = WL.rng(43)
    M, N, K = 77, 384, 512
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, "uint4_zp", N, K)
    d, packed = G.pack(w)
    qg.force_config(128, 1)                 # the same token tile and no split in both calls
    try:
        y_moe = _run_moe([w], x, [0, M])
        y_dense = G.to_f64(qg.w4a16(d, packed, G.bf16_tensor(x)))
    finally:
        qg.force_config(0, 0)
    np.testing.assert_array_equal(y_moe, y_dense)


def test_moe_rows_outside_groups_untouched():
    """Rows before offsets[0] and after offsets[E] are not written."""
    r = WL.rng(44)
    counts = [9, 0, 20]
    off = _offsets(counts) + 5
    R = int(off[-1]) + 7
    N, K = 256, 256
    x = WL.gen_x(r, R, K)
    ws = [WL.gen_weights(r, "mxfp4", N, K) for _ in counts]
    y = _run_moe(ws, x, off, out_fill=3.0)
    assert np.all(y[:5] == 3.0) and np.all(y[int(off[-1]):] == 3.0)
    ref = oracle.moe_grouped(F_bits(x)[5:int(off[-1])], off - 5, _experts_a16(ws))
    _assert_close(y[5:int(off[-1])], ref, TOL_A16)


@pytest.mark.parametrize("afmt", ["fp8", "fp8n"])
@pytest.mark.parametrize("stream_k", [False, True])
def test_moe_a8_parity(stream_k, afmt):
    r = WL.rng(45)
    counts = [12, 0, 41, 200, 1]
    off = _offsets(counts)
    R = int(off[-1])
    N, K = 512, 1024
    x = WL.gen_x(r, R, K, outliers=True)
    xq, s = oracle.quant_act_fp8(x)
    ws = [WL.gen_weights(r, "mxfp4", N, K) for _ in counts]
    from oracle import formats as F
    ref = oracle.moe_grouped(F.e4m3_to_float(xq), off, _experts_exact(ws), tok_scale=s)
    _assert_close(_run_moe(ws, xq, off, afmt=afmt, tok_scale=s, stream_k=stream_k, calls=2),
                  ref, TOL_A8)


@pytest.mark.parametrize("T", [1, 128])
def test_moe_router_workload_sampled(T):
    """The DeepSeek-V3-like layer's gate_up GEMM (E = 256 MXFP4 experts of 4096 x 7168)
    at T tokens routed top-8 with the skewed logits, in the launch configuration the
    benchmark times (with the MoE workspace): up to 32 sampled rows (each against its own
    expert) plus every row of the two largest experts."""
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    case = WL.moe_case(T, seed=0, skewed=True)
    E, N, K = WL.MOE_E, 2 * WL.MOE_INTER, WL.MOE_HIDDEN
    off = np.asarray(case.offsets, dtype=np.int64)
    R = int(off[-1])
    r = WL.rng(46)
    rows = set(int(v) for v in r.choice(R, size=min(32, R), replace=False))
    for e in np.argsort(-np.diff(off), kind="stable")[:2]:
        rows.update(range(int(off[e]), int(off[e + 1])))
    rows = sorted(rows)
    expert_of = np.searchsorted(off, np.asarray(rows), side="right") - 1
    d = qg.WeightDesc("mxfp4", N, K, 32)
    nb = qg.packed_bytes(d)
    packed = torch.empty(nb * E, dtype=torch.uint8, device="cuda")
    xf = F_bits(case.x_bits)
    ref = np.zeros((len(rows), N))
    for e, w in enumerate(WL.iter_moe_weights(E, N, K, seed=0)):
        qg.repack(d, G.u8_tensor(w.codes), G.u8_tensor(w.scales), None,
                  out=packed[e * nb:(e + 1) * nb])
        mine = np.nonzero(expert_of == e)[0]
        if len(mine):
            W = oracle.dequant(w.wfmt, w.group, w.codes, w.scales)
            ref[mine] = oracle.gemm(xf[[rows[i] for i in mine]], W)
    X = G.bf16_tensor(case.x_bits)
    y = qg.moe_grouped(d, packed, E, X, torch.tensor(off.astype(np.int32), device="cuda"),
                       ws=qg.moe_workspace(d, E, R))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    y = G.to_f64(y)
    _assert_close(y[rows], ref, TOL_A16)


# ------------------------------------------------------------------------- indexed

def _run_moe_indexed(ws, x_bits, offsets, row_index, afmt="bf16", tok_scale=None, stream_k=False):
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    d, packed = _pack_experts(ws, afmt)
    off = torch.tensor(np.asarray(offsets, dtype=np.int32), device="cuda")
    idx = torch.tensor(np.asarray(row_index, dtype=np.int32), device="cuda")
    R = idx.numel()
    wsp = qg.moe_workspace(d, len(ws), R) if stream_k else None
    out = torch.full((R, ws[0].N), 5.0, dtype=torch.bfloat16, device="cuda")
    for _ in range(2):              # the second call checks that the workspace came back clean
        if afmt == "bf16":
            y = qg.moe_indexed(d, packed, len(ws), G.bf16_tensor(x_bits), off, idx, out=out, ws=wsp)
        else:
            ts = torch.from_numpy(np.asarray(tok_scale, dtype=np.float32)).cuda()
            y = qg.moe_indexed(d, packed, len(ws), G.u8_tensor(x_bits), off, idx, tok_scale=ts,
                               out=out, ws=wsp)
        torch.cuda.synchronize()
        assert qg.device_status(clear=True) == 0
    return G.to_f64(y)


@pytest.mark.parametrize("stream_k", [False, True])
@pytest.mark.parametrize("afmt", ["bf16", "fp8", "fp8n"])
def test_moe_indexed_router(afmt, stream_k):
    """Routed tokens gathered from X in token order (padding positions index -1), against
    the oracle; FP8 rows take the scale of the row they come from."""
    case = WL.moe_case(T=40, seed=5, E=8, topk=2, hidden=256, inter=64)
    r = WL.rng(47)
    ws = [WL.gen_weights(r, "mxfp4", 256, 256) for _ in range(8)]
    idx = case.token_of_row.astype(np.int32)
    if afmt == "bf16":
        x = case.x_tok_bits
        ref = oracle.moe_indexed(F_bits(x), case.offsets, idx, _experts_a16(ws))
        _assert_close(_run_moe_indexed(ws, x, case.offsets, idx, stream_k=stream_k), ref, TOL_A16)
    else:
        from oracle import formats as F
        xq, s = oracle.quant_act_fp8(WL.gen_x(WL.rng(48), case.T, 256, outliers=True))
        ref = oracle.moe_indexed(F.e4m3_to_float(xq), case.offsets, idx, _experts_exact(ws),
                                 tok_scale=s)
        y = _run_moe_indexed(ws, xq, case.offsets, idx, afmt=afmt, tok_scale=s, stream_k=stream_k)
        _assert_close(y, ref, TOL_A8)


@pytest.mark.parametrize("wfmt,afmt", [("mxfp4", "bf16"), ("uint4_zp", "bf16"), ("mxfp4", "fp8"),
                                       ("mxfp4", "fp8n")])
@pytest.mark.parametrize("copy", [False, True])
def test_moe_indexed_many_rows(wfmt, afmt, copy):
    """Indexed calls of 256 rows or more (here over 2048): with the indexed workspace the rows are gathered
    into it first and the grouped kernel runs on the copy; with a forced token tile the
    gathering kernel runs instead.  Both against the oracle, twice on one workspace."""
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    case = WL.moe_case(T=320, seed=9, E=16, topk=8, hidden=512, inter=64)
    r = WL.rng(49)
    ws = [WL.gen_weights(r, wfmt, 256, 512) for _ in range(16)]
    idx = case.token_of_row.astype(np.int32)
    R, T = len(idx), case.T
    assert R >= 2048
    fp8 = afmt != "bf16"
    d, packed = _pack_experts(ws, afmt)
    off = torch.tensor(np.asarray(case.offsets, dtype=np.int32), device="cuda")
    it = torch.tensor(idx, device="cuda")
    wsp = qg.moe_indexed_workspace(d, 16, T, R, fp8=fp8)
    if fp8:
        from oracle import formats as F
        xq, s = oracle.quant_act_fp8(WL.gen_x(WL.rng(50), T, 512, outliers=True))
        ref = oracle.moe_indexed(F.e4m3_to_float(xq), case.offsets, idx, _experts_exact(ws),
                                 tok_scale=s)
        X = G.u8_tensor(xq)
        ts = torch.from_numpy(s).cuda()
    else:
        x = case.x_tok_bits
        ref = oracle.moe_indexed(F_bits(x), case.offsets, idx, _experts_a16(ws))
        X = G.bf16_tensor(x)
        ts = None
    out = torch.empty(R, 256, dtype=torch.bfloat16, device="cuda")
    if not copy:
        qg.force_config(32, 0)       # a forced token tile keeps the in-kernel gather
    try:
        for _ in range(2):
            out.fill_(float("nan"))
            y = qg.moe_indexed(d, packed, 16, X, off, it, tok_scale=ts, out=out, ws=wsp)
            torch.cuda.synchronize()
            assert qg.device_status(clear=True) == 0
            valid = idx >= 0
            _assert_close(G.to_f64(y)[valid], ref[valid], TOL_A8 if fp8 else TOL_A16)
    finally:
        qg.force_config(0, 0)


def test_moe_indexed_nvfp4():
    """Indexed rows with NVFP4 experts, each with its own per-tensor scale, with and without
    stream-K (K blocks enough to cut the leftover tiles)."""
    r = WL.rng(54)
    T, N, K = 9, 7168, 3072
    counts = [1, 1, 2, 1, 1, 1, 1, 1]
    off = _offsets(counts)
    idx = r.permutation(T)[:int(off[-1])].astype(np.int32)
    x = WL.gen_x(r, T, K)
    ws = [WL.gen_weights(r, "nvfp4", N, K) for _ in counts]
    assert len(set(w.global_scale for w in ws)) == len(ws)
    ref = oracle.moe_indexed(F_bits(x), off, idx, _experts_a16(ws))
    for sk in (False, True):
        _assert_close(_run_moe_indexed(ws, x, off, idx, stream_k=sk), ref, TOL_A16)


@pytest.mark.parametrize("tile", [16, 32, 64])
def test_moe_indexed_every_tile(tile):
    """Arbitrary gathers: repeated rows, rows in any order, padding, empty experts and
    blocks longer than one tile, for each token tile a gathered tile can have."""
    import quantized_weight_gemm_gb300 as qg
    r = WL.rng(49)
    T, N, K = 37, 384, 512
    counts = [0, 9, 1, 40, 0, 3, 17, 2]
    off = _offsets(counts)
    R = int(off[-1])
    idx = r.integers(-1, T, size=R).astype(np.int32)          # includes -1 (padding)
    x = WL.gen_x(r, T, K)
    ws = [WL.gen_weights(r, "uint4_zp", N, K) for _ in counts]
    ref = oracle.moe_indexed(F_bits(x), off, idx, _experts_a16(ws))
    qg.force_config(tile, 0)
    try:
        y = _run_moe_indexed(ws, x, off, idx)
    finally:
        qg.force_config(0, 0)
    _assert_close(y, ref, TOL_A16)
    assert np.all(y[idx < 0] == 0)


def test_moe_indexed_stream_k():
    """Enough leftover tiles for the kernel to cut them over several CTAs (448 gathered
    tiles of 16 rows: two whole rounds and 144 tiles of 24 K blocks cut)."""
    r = WL.rng(50)
    T, N, K = 12, 7168, 3072
    counts = [1, 1, 2, 1, 1, 1, 1, 1]
    off = _offsets(counts)
    idx = r.permutation(T)[:int(off[-1])].astype(np.int32)
    x = WL.gen_x(r, T, K)
    ws = [WL.gen_weights(r, "mxfp4", N, K) for _ in counts]
    ref = oracle.moe_indexed(F_bits(x), off, idx, _experts_a16(ws))
    _assert_close(_run_moe_indexed(ws, x, off, idx, stream_k=True), ref, TOL_A16)


@pytest.mark.parametrize("tile", [16, 64])
def test_moe_indexed_ragged_k_and_stride(tile):
    """K = 608 ends inside an activation slot (512 K for 16-row tiles, 256 for 64), and X is a
    view into wider rows whose extra columns hold NaN: the gathered copies must stop at K
    and zero-fill the rest of the slot."""
    import quantized_weight_gemm_gb300 as qg
    from tests import gpu_util as G
    r = WL.rng(52)
    T, N, K = 29, 256, 608
    counts = [5, 0, 30, 11]
    off = _offsets(counts)
    idx = r.integers(-1, T, size=int(off[-1])).astype(np.int32)
    x = WL.gen_x(r, T, K)
    ws = [WL.gen_weights(r, "mxfp4", N, K) for _ in counts]
    ref = oracle.moe_indexed(F_bits(x), off, idx, _experts_a16(ws))
    wide = torch.full((T, K + 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    wide[:, :K] = G.bf16_tensor(x)
    d, packed = _pack_experts(ws)
    qg.force_config(tile, 0)
    try:
        y = qg.moe_indexed(d, packed, len(ws), wide[:, :K],
                           torch.tensor(off, dtype=torch.int32, device="cuda"),
                           torch.tensor(idx, device="cuda"))
        torch.cuda.synchronize()
        assert qg.device_status(clear=True) == 0
    finally:
        qg.force_config(0, 0)
    y = G.to_f64(y)
    assert np.all(np.isfinite(y))
    _assert_close(y, ref, TOL_A16)


def test_moe_indexed_index_past_end():
    """A row index at or past T is reported in the device status word (BAD_VALUE) and its
    row reads as zeros; the other rows are unaffected."""
    import quantized_weight_gemm_gb300 as qg
    from tests import gpu_util as G
    r = WL.rng(53)
    T, N, K = 10, 256, 256
    counts = [3, 4]
    off = _offsets(counts)
    idx = np.array([0, 9, T, 2, T + 1000, -1, 5], dtype=np.int32)
    x = WL.gen_x(r, T, K)
    ws = [WL.gen_weights(r, "mxfp4", N, K) for _ in counts]
    ok_idx = np.where(idx < T, idx, -1).astype(np.int32)
    ref = oracle.moe_indexed(F_bits(x), off, ok_idx, _experts_a16(ws))
    d, packed = _pack_experts(ws)
    qg.device_status(clear=True)
    y = qg.moe_indexed(d, packed, len(ws), G.bf16_tensor(x),
                       torch.tensor(off, dtype=torch.int32, device="cuda"),
                       torch.tensor(idx, device="cuda"))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 9          # QGEMM_ERR_BAD_VALUE
    y = G.to_f64(y)
    assert np.all(y[idx >= T] == 0)
    _assert_close(y, ref, TOL_A16)


def test_moe_batch_invariant():
    """With the flag, expert 0's rows are the same bits whatever the other experts' loads
    (the default token tile and stream-K follow R / E), and the indexed call refuses it."""
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    r = WL.rng(55)
    N, K = 256, 2048
    ws = [WL.gen_weights(r, "mxfp4", N, K) for _ in range(4)]
    x0 = WL.gen_x(r, 40, K)
    codes = G.u8_tensor(_stack(ws, "codes"))
    sc = G.u8_tensor(_stack(ws, "scales"))
    d = qg.WeightDesc("mxfp4", N, K, 32, batch_invariant=True)
    packed = qg.repack(d, codes, sc, None, num_experts=4)
    outs = []
    for counts in ([40, 0, 0, 0], [40, 300, 7, 900], [40, 1, 1, 1]):
        off = _offsets(counts)
        R = int(off[-1])
        xr = np.concatenate([x0, WL.gen_x(r, R - 40, K)]) if R > 40 else x0
        wsp = qg.moe_workspace(d, 4, R)
        y = qg.moe_grouped(d, packed, 4, G.bf16_tensor(xr),
                           torch.tensor(off, dtype=torch.int32, device="cuda"), ws=wsp)
        outs.append(G.bf16_bits_of(y)[:40])
        ref = oracle.moe_grouped(F_bits(xr), off, _experts_a16(ws))
        _assert_close(G.to_f64(y), ref, TOL_A16)
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])
    with pytest.raises(qg.QGemmError):
        qg.moe_indexed(d, packed, 4, G.bf16_tensor(x0),
                       torch.tensor([0, 40, 40, 40, 40], dtype=torch.int32, device="cuda"),
                       torch.arange(40, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0


def test_moe_indexed_refuses_wide_tiles():
    import quantized_weight_gemm_gb300 as qg
    r = WL.rng(51)
    ws = [WL.gen_weights(r, "mxfp4", 256, 256) for _ in range(2)]
    qg.force_config(128, 0)
    try:
        with pytest.raises(qg.QGemmError):
            _run_moe_indexed(ws, WL.gen_x(r, 4, 256), [0, 2, 4], [0, 1, 2, 3])
    finally:
        qg.force_config(0, 0)
