"""Repack + register decode, bit-exact against the oracle's RNE_bf16(dequant(W)).

The GPU decodes the packed form through the same device functions the GEMM kernels use;
every bit must match (+0 and -0 compare equal), across formats, group sizes, ragged N and
K, and extreme E8M0 exponents."""
import numpy as np
import pytest
import torch

import oracle
from oracle import formats as F
import workloads as WL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from quantized_weight_gemm_gb300 import build
    build.build()
    import quantized_weight_gemm_gb300 as qg
    qg.device_status(clear=True)
    yield
    assert qg.device_status(clear=True) == 0


def _check(w, afmt="bf16"):
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    d, packed = G.pack(w, afmt)
    got = G.to_f64(qg.dequant_debug(d, packed))
    ref = F.round_to_bf16(oracle.dequant(w.wfmt, w.group, w.codes, w.scales, w.zeros,
                                         w.global_scale))
    torch.cuda.synchronize()
    assert qg.device_status(clear=True) == 0
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    if not np.all(same):
        bad = np.argwhere(~same)[:5]
        raise AssertionError(f"{(~same).sum()} mismatches, e.g. {[(tuple(b), got[tuple(b)], ref[tuple(b)]) for b in bad]}")


@pytest.mark.parametrize("wfmt,group", [("int4_sym", 128), ("uint4_zp", 128), ("int4_sym", 32),
                                        ("uint4_zp", 32), ("uint4_zp", 64), ("uint4_zp", 256),
                                        ("mxfp4", 32), ("mxint4", 32), ("nvfp4", 16)])
@pytest.mark.parametrize("N,K", [(256, 512), (300, 768), (1, 256), (130, 96)])
def test_repack_roundtrip_bitexact(wfmt, group, N, K):
    if K % group:
        pytest.skip("K not a multiple of the group")
    r = WL.rng(11)
    w = WL.gen_weights(r, wfmt, N, K, group=group, zp_lo=0, zp_hi=15)
    _check(w)


@pytest.mark.parametrize("afmt", ["fp8", "fp8n"])
@pytest.mark.parametrize("N,K", [(256, 512), (200, 160)])
def test_repack_roundtrip_fp8_layout(N, K, afmt):
    w = WL.gen_weights(WL.rng(12), "mxfp4", N, K)
    _check(w, afmt=afmt)


def test_mxfp4_all_exponents():
    # every E8M0 exponent 0..254 (two-step scaling above 128, subnormal results below)
    r = WL.rng(13)
    N, K = 255, 64
    w = WL.gen_weights(r, "mxfp4", N, K)
    w.scales[:] = np.arange(255, dtype=np.uint8)[:, None]
    _check(w)
    _check(w, afmt="fp8")
    _check(w, afmt="fp8n")


def test_mxint4_all_exponents():
    """Every E8M0 exponent 0..254: the subnormal factor 2^-127 at 0, overflow to infinity
    at the top, exactly as RNE_bf16 of the exact weight."""
    r = WL.rng(16)
    w = WL.gen_weights(r, "mxint4", 255, 64)
    w.scales[:] = np.arange(255, dtype=np.uint8)[:, None]
    _check(w)


@pytest.mark.parametrize("g", [1.0, 0.37, 2.0 ** -20])
def test_nvfp4_all_scales(g):
    """Every E4M3 scale code but NaN (either sign, subnormals included) with every e2m1
    code, times a per-tensor scale: one rounding of the exact product."""
    r = WL.rng(17)
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    w = WL.gen_weights(r, "nvfp4", len(codes), 64)
    w.scales[:] = codes[:, None]
    w.global_scale = float(np.float32(g))
    _check(w)


def test_int4_scale_extremes():
    r = WL.rng(14)
    w = WL.gen_weights(r, "uint4_zp", 128, 256, group=128, zp_lo=0, zp_hi=15)
    # subnormal, tiny, huge and negative bf16 scales
    vals = np.array([1e-40, 2.0 ** -126, 3.0e38, -0.75, 1.0, 65504.0, -2.0 ** -130, 1.5],
                    dtype=np.float32)
    w.scales[:] = WL.to_bf16_bits(vals[np.arange(w.scales.size) % len(vals)].reshape(w.scales.shape))
    _check(w)


def test_repack_rejects_bad_values():
    from tests import gpu_util as G
    import quantized_weight_gemm_gb300 as qg
    w = WL.gen_weights(WL.rng(15), "mxfp4", 128, 64)
    w.scales[3, 1] = 255
    G.pack(w)
    assert qg.device_status(clear=True) == 9
    w = WL.gen_weights(WL.rng(15), "uint4_zp", 128, 128, group=128)
    w.zeros[0, 0] = 16
    G.pack(w)
    assert qg.device_status(clear=True) == 9
    for nan in (0x7F, 0xFF):                                # E4M3 NaN scales
        w = WL.gen_weights(WL.rng(15), "nvfp4", 128, 64)
        w.scales[5, 2] = nan
        G.pack(w)
        assert qg.device_status(clear=True) == 9
