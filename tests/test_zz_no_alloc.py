"""qgemm_w4a16_noalloc: the W4A16 GEMM for callers that cannot allocate a workspace.

Such callers (a framework whose allocator owns all device memory, or a latency-critical
path that must avoid cudaMalloc) get the split-K scratch from a fixed array inside the
library instead of a workspace argument.  This file is collected last on purpose.  Its
checks, through the C ABI:
  * two calls in a row of the no-alloc entry point give the same bits as qgemm_w4a16 with
    a workspace (both run the same schedule) and pass the W4A16 bar against the oracle,
    for uniform K cuts and for stream-K;
  * a call needs only what its own schedule uses, whatever smaller M would need (above
    M = 1024 nothing is cut below K = 16384: INT4 with BF16 scales needs its FP16
    activation copy, MXFP4 nothing; with longer K the stream-K schedule there gives way
    to whole tiles when its partial sums do not fit the array);
  * a call whose schedule needs more scratch than the built-in array is refused with
    QGEMM_ERR_WORKSPACE.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as WL

pytestmark = pytest.mark.gpu

TOL = 8e-3
SCRATCH_BYTES = 8 * 1024 * 1024


@pytest.fixture(scope="module")
def qg():
    from quantized_weight_gemm_gb300 import build
    build.build()
    import quantized_weight_gemm_gb300 as q
    q.force_config(0, 0)
    q.device_status(clear=True)
    yield q
    q.force_config(0, 0)


def _noalloc(qg, d, packed, X, M, N):
    cd = d.c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = qg.lib().qgemm_w4a16_noalloc(ctypes.byref(cd), ctypes.c_void_p(packed.data_ptr()),
                                      ctypes.c_void_p(X.data_ptr()), M, X.stride(0), None,
                                      ctypes.c_void_p(y.data_ptr()), y.stride(0), stream)
    return st, y


@pytest.mark.parametrize("wfmt,M,N,K,cut", [("uint4_zp", 16, 4096, 4096, "any"),
                                            ("mxfp4", 1, 4096, 7168, "any"),
                                            ("int4_sym", 64, 1024, 4096, "any"),
                                            ("uint4_zp", 1, 28672, 8192, "stream-k")])
def test_noalloc_matches_workspace_entry_point(qg, wfmt, M, N, K, cut):
    from tests import gpu_util as G
    r = WL.rng(31)
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, wfmt, N, K, group=32 if wfmt == "mxfp4" else 128)
    d, packed = G.pack(w)
    p = qg.plan(d, M)
    assert p["splits"] > 1 or p["sk_tiles"] > 0    # this schedule cuts tiles: it uses scratch
    if cut == "stream-k":
        assert p["sk_tiles"] > 0 and p["max_contrib"] > 1
    X = G.bf16_tensor(x)
    ref_dev = G.bf16_bits_of(qg.w4a16(d, packed, X))
    torch.cuda.synchronize()
    ref = oracle.w4a16(x, w.wfmt, w.group, w.codes, w.scales, w.zeros)
    for _ in range(2):                            # the scratch is reused by the second call
        st, y = _noalloc(qg, d, packed, X, M, N)
        assert st == 0
        torch.cuda.synchronize()
        assert qg.device_status(clear=True) == 0
        np.testing.assert_array_equal(G.bf16_bits_of(y), ref_dev)
        ok, worst = oracle.tolerance_ok(G.to_f64(y), ref, TOL)
        assert ok, f"worst error / bound = {worst:.3f}"


@pytest.mark.parametrize("wfmt,N,K,M", [("uint4_zp", 28672, 3072, 1100), ("mxfp4", 4096, 7168, 8192)])
def test_noalloc_sized_by_its_own_schedule(qg, wfmt, N, K, M):
    """Above M = 1024 the default schedule cuts no tile, so a call needs only what its own
    schedule uses -- INT4 with BF16 scales its FP16 activation copy (6.4 MiB here, while
    a smaller M's cut schedule would need more than the array), MXFP4 nothing at all."""
    from tests import gpu_util as G
    r = WL.rng(33)
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, wfmt, N, K)
    d, packed = G.pack(w)
    p = qg.plan(d, M)
    assert p["splits"] == 1 and p["sk_tiles"] == 0
    assert qg.act_copy_bytes(d, M) <= SCRATCH_BYTES
    if wfmt == "uint4_zp":
        assert qg.workspace_bytes(d, M) > SCRATCH_BYTES
    X = G.bf16_tensor(x)
    st, y = _noalloc(qg, d, packed, X, M, N)
    assert st == 0
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    ref_dev = qg.w4a16(d, packed, X)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), ref_dev.view(torch.int16))


def test_noalloc_refuses_oversized_plan(qg):
    from tests import gpu_util as G
    w = WL.gen_weights(WL.rng(32), "uint4_zp", 28672, 1024)
    d, packed = G.pack(w)
    X = torch.zeros(256, 1024, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(256, 28672, dtype=torch.bfloat16, device="cuda")
    qg.force_config(128, 4)                      # 2 x 224 tiles x 4 FP32 partials >> 8 MiB
    try:
        assert qg.workspace_bytes(d, 256) > SCRATCH_BYTES
        cd = d.c()
        st = qg.lib().qgemm_w4a16_noalloc(ctypes.byref(cd), ctypes.c_void_p(packed.data_ptr()),
                                          ctypes.c_void_p(X.data_ptr()), 256, 1024, None,
                                          ctypes.c_void_p(Y.data_ptr()), 28672, None)
        assert st == 4
    finally:
        qg.force_config(0, 0)


def test_noalloc_long_k_large_m_keeps_whole_tiles(qg):
    """K >= 16384 above M = 1024: the default schedule runs stream-K, whose partial sums do
    not fit the array, so the no-alloc call runs whole tiles instead of refusing -- the
    same bits as qgemm_w4a16 with a workspace too small for stream-K."""
    from tests import gpu_util as G
    N, K, M = 4096, 16384, 2048
    r = WL.rng(35)
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, "mxfp4", N, K)
    d, packed = G.pack(w)
    p = qg.plan(d, M)
    assert p["sk_tiles"] > 0 and p["max_contrib"] > 1
    assert qg.workspace_bytes(d, M) > SCRATCH_BYTES
    X = G.bf16_tensor(x)
    st, y = _noalloc(qg, d, packed, X, M, N)
    assert st == 0
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    ref_dev = qg.w4a16(d, packed, X, ws=small)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), ref_dev.view(torch.int16))
