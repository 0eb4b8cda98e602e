"""The kernels' bounded waits: a wait that runs into its time limit ends the call with
QGEMM_ERR_TIMEOUT in the status word, and the context stays usable.

The failure is made without faulting anything: under qgemm_debug_stall the activation
producer of each CTA never issues its first load (nothing is in flight for that slot, and
no wait is removed), so the MMA issuers' wait for it, and then every other role's, gives
up after the limit set for the test; the kernel waits for the copies it did issue,
releases its tensor memory and returns.  A normal call afterwards, in the same process,
must pass parity.  The pages' counterpart: failures isolated so that inference survives
them (the Chinese release notes, v0.1.1)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as WL

pytestmark = pytest.mark.gpu

QGEMM_ERR_TIMEOUT = 7


@pytest.fixture(scope="module")
def qg():
    from quantized_weight_gemm_gb300 import build
    build.build()
    import quantized_weight_gemm_gb300 as q
    q.force_config(0, 0)
    q.debug_stall(0, 0)
    q.device_status(clear=True)
    yield q
    q.debug_stall(0, 0)
    q.force_config(0, 0)


@pytest.mark.parametrize("wfmt,M,N,K", [("uint4_zp", 16, 1024, 1024), ("mxfp4", 300, 512, 512)])
def test_wait_limit_ends_the_call(qg, wfmt, M, N, K):
    from tests import gpu_util as G
    r = WL.rng(40)
    x = WL.gen_x(r, M, K)
    w = WL.gen_weights(r, wfmt, N, K)
    d, packed = G.pack(w)
    X = G.bf16_tensor(x)
    qg.debug_stall(1, 20)                       # 20 ms wait limit
    try:
        qg.w4a16(d, packed, X)                  # launches; the kernel gives up on the device
        torch.cuda.synchronize()
    finally:
        qg.debug_stall(0, 0)
    assert qg.device_status(clear=True) == QGEMM_ERR_TIMEOUT
    assert qg.device_status(clear=True) == 0    # the status word was cleared
    # the same process, the same buffers: a normal call passes parity
    y = G.to_f64(qg.w4a16(d, packed, X))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    ref = oracle.w4a16(x, w.wfmt, w.group, w.codes, w.scales, w.zeros)
    ok, worst = oracle.tolerance_ok(y, ref, 8e-3)
    assert ok, f"worst error / bound = {worst:.3f}"
