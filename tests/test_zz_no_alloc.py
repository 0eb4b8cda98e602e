"""qgemm_w4a16_noalloc: the W4A16 GEMM for callers that cannot allocate a workspace.

Such callers (a framework whose allocator owns all device memory, or a latency-critical
path that must avoid cudaMalloc) get the split-K scratch from a fixed array inside the
library instead of a workspace argument.  This file is collected last on purpose.  Its
checks: through the C ABI, two calls in a row of the no-alloc entry point agree with
qgemm_w4a16 (given a normal workspace) within the W4A16 tolerance, and a call whose plan
needs more scratch than the built-in array is refused with QGEMM_ERR_WORKSPACE.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as WL

pytestmark = pytest.mark.gpu

TOL = 8e-3
SCRATCH_BYTES = 8 * 1024 * 1024


def _close(y, ref):
    y = y.double().cpu().numpy()
    ref = ref.double().cpu().numpy()
    rms = np.sqrt(np.mean(ref * ref))
    return np.all(np.abs(y - ref) <= TOL * np.maximum(np.abs(ref), rms))


@pytest.fixture(scope="module")
def qg():
    from quantized_weight_gemm_gb300 import build
    build.build()
    import quantized_weight_gemm_gb300 as q
    q.force_config(0, 0)
    q.device_status(clear=True)
    yield q
    q.force_config(0, 0)


@pytest.mark.parametrize("wfmt,M,N,K", [("uint4_zp", 16, 4096, 4096), ("mxfp4", 1, 4096, 7168),
                                        ("int4_sym", 64, 1024, 2048)])
def test_noalloc_matches_workspace_entry_point(qg, wfmt, M, N, K):
    from tests import gpu_util as G
    r = WL.rng(31)
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, wfmt, N, K, group=32 if wfmt == "mxfp4" else 128)
    d, packed = G.pack(w)
    assert qg.workspace_bytes(d, M) > 0          # this case runs split-K, i.e. uses scratch
    X = G.bf16_tensor(x)
    ref = qg.w4a16(d, packed, X)
    L = qg.lib()
    cd = d.c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):                            # the scratch is reused by the second call
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = L.qgemm_w4a16_noalloc(ctypes.byref(cd), ctypes.c_void_p(packed.data_ptr()),
                                   ctypes.c_void_p(X.data_ptr()), M, X.stride(0), None,
                                   ctypes.c_void_p(y.data_ptr()), y.stride(0), stream)
        assert st == 0
        torch.cuda.synchronize()
        assert qg.device_status(clear=True) == 0
        assert _close(y, ref)


def test_noalloc_refuses_oversized_plan(qg):
    from tests import gpu_util as G
    w = WL.gen_weights(WL.rng(32), "uint4_zp", 28672, 1024)
    d, packed = G.pack(w)
    X = torch.zeros(256, 1024, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(256, 28672, dtype=torch.bfloat16, device="cuda")
    qg.force_config(256, 4)                      # 256 x 28672 fp32 partials > 8 MiB
    try:
        assert qg.workspace_bytes(d, 256) > SCRATCH_BYTES
        cd = d.c()
        st = qg.lib().qgemm_w4a16_noalloc(ctypes.byref(cd), ctypes.c_void_p(packed.data_ptr()),
                                          ctypes.c_void_p(X.data_ptr()), 256, 1024, None,
                                          ctypes.c_void_p(Y.data_ptr()), 28672, None)
        assert st == 4
    finally:
        qg.force_config(0, 0)
