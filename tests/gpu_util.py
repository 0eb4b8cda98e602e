"""Helpers for the GPU parity tests: numpy <-> torch marshalling and case builders."""
import numpy as np
import torch

import quantized_weight_gemm_gb300 as qg

DEV = "cuda"


def bf16_tensor(bits):
    """uint16 bf16 bit patterns (numpy) -> torch.bfloat16 on the GPU."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def u8_tensor(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(DEV)


def scales_tensor(w):
    if w.scales.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(w.scales).view(np.int16)).to(DEV)
    return u8_tensor(w.scales)


def to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def bf16_bits_of(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def desc_of(w, afmt="bf16"):
    return qg.WeightDesc(w.wfmt, w.N, w.K, w.group, afmt)


def pack(w, afmt="bf16"):
    d = desc_of(w, afmt)
    z = None if w.zeros is None else u8_tensor(w.zeros)
    return d, qg.repack(d, u8_tensor(w.codes), scales_tensor(w), z, global_scale=w.global_scale)


def ref_bf16_weights(x_bits, w, chan_scale=None):
    """The product on the weights rounded to BF16 (the arithmetic of a kernel that scales
    its weights before a BF16 tensor core), for reporting beside the exact reference."""
    import oracle
    from oracle import formats as F
    W = oracle.dequant_bf16(w.wfmt, w.group, w.codes, w.scales, w.zeros)
    y = oracle.gemm(F.bf16_bits_to_float(x_bits), W, chan_scale=chan_scale)
    return y * np.float64(np.float32(w.global_scale))


def log_parity(tag, y, ref, tol, ref_bf16=None):
    """Append the worst error/bound against the exact reference (and, when given, against
    the BF16-weight product) to the JSON-lines file named by QGEMM_PARITY_LOG, if set."""
    import json
    import os
    import oracle
    path = os.environ.get("QGEMM_PARITY_LOG")
    if not path:
        return
    rec = {"case": tag, "tol": tol, "worst_exact": oracle.tolerance_ok(y, ref, tol)[1],
           "outputs": int(np.asarray(ref).size)}
    if ref_bf16 is not None:
        rec["worst_bf16_weights"] = oracle.tolerance_ok(y, ref_bf16, tol)[1]
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")
