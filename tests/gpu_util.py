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
