"""Python binding of the qgemm C ABI (include/qgemm.h): argument marshalling only.

Every computation runs in libqgemm.so's sm_103a kernels; this module only checks
tensor dtypes/devices, passes raw pointers and the current CUDA stream, and turns status
codes into exceptions.  There is no fallback: if the library is missing, every call
raises.
"""
import ctypes
import os
from dataclasses import dataclass

import torch

__all__ = [
    "QGemmError", "WeightDesc", "lib", "lib_path", "packed_bytes", "repack", "workspace_bytes",
    "w4a16", "w4a8", "quant_act_fp8", "moe_grouped", "dequant_debug", "device_status",
    "force_config", "plan", "moe_workspace_bytes", "moe_workspace", "moe_indexed_workspace_bytes",
    "moe_indexed_workspace", "host_staging_bytes",
    "host_staging", "w4a16_host", "moe_indexed", "check_desc", "WFMT", "AFMT", "EXPORTS",
    "debug_stall", "act_copy_bytes", "w4a4", "quant_act_mxfp4",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_lib", "libqgemm.so")

WFMT = {"int4_sym": 0, "uint4_zp": 1, "mxfp4": 2, "mxint4": 3, "nvfp4": 4}
SDTYPE = {"int4_sym": 0, "uint4_zp": 0, "mxfp4": 1, "mxint4": 1, "nvfp4": 2}   # BF16, E8M0, E4M3
AFMT = {"bf16": 0, "fp8": 1, "mxfp4": 2, "fp8n": 3}   # fp8n: W4A8 on FP4 tensor-core operands
EXPORTS = ("qgemm_version", "qgemm_status_str", "qgemm_check_desc", "qgemm_packed_bytes",
           "qgemm_repack", "qgemm_workspace_bytes", "qgemm_w4a16", "qgemm_quant_act_fp8",
           "qgemm_w4a8", "qgemm_moe_grouped", "qgemm_dequant_debug", "qgemm_device_status",
           "qgemm_force_config", "qgemm_w4a16_noalloc", "qgemm_plan",
           "qgemm_moe_workspace_bytes", "qgemm_host_staging_bytes", "qgemm_w4a16_host",
           "qgemm_moe_indexed", "qgemm_repack_scaled", "qgemm_debug_stall",
           "qgemm_act_copy_bytes", "qgemm_w4a4", "qgemm_quant_act_mxfp4",
           "qgemm_moe_indexed_workspace_bytes")

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "alignment", 4: "workspace",
          5: "bad packed", 6: "cuda error", 7: "timeout", 8: "no device", 9: "bad value"}


class QGemmError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = int(status)
        super().__init__(f"qgemm: {what}: status {status} ({STATUS.get(int(status), '?')})")


class _WDesc(ctypes.Structure):
    _fields_ = [("wfmt", ctypes.c_int32), ("sdtype", ctypes.c_int32),
                ("group_size", ctypes.c_int32), ("has_zp", ctypes.c_int32),
                ("afmt", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


@dataclass(frozen=True)
class WeightDesc:
    """One quantized weight matrix [N, K]: format, group size and activation format.
    batch_invariant: every call runs one schedule for all M (QGEMM_FLAG_BATCH_INVARIANT)."""
    wfmt: str
    N: int
    K: int
    group: int = 128
    afmt: str = "bf16"
    batch_invariant: bool = False

    def c(self):
        w = WFMT[self.wfmt]
        return _WDesc(w, SDTYPE[self.wfmt], self.group,
                      1 if self.wfmt == "uint4_zp" else 0, AFMT[self.afmt],
                      1 if self.batch_invariant else 0, self.N, self.K)


_lib = None


def lib_path():
    return _LIB_PATH


def lib():
    """Load libqgemm.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"libqgemm.so not built ({_LIB_PATH}); run "
                           "`python -m quantized_weight_gemm_gb300.build`")
    L = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    I32, I64, SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    D = ctypes.POINTER(_WDesc)
    sigs = {
        "qgemm_version": (I32, []),
        "qgemm_status_str": (ctypes.c_char_p, [ctypes.c_int]),
        "qgemm_check_desc": (ctypes.c_int, [D]),
        "qgemm_packed_bytes": (SZ, [D]),
        "qgemm_repack": (ctypes.c_int, [D, P, P, P, P, P]),
        "qgemm_repack_scaled": (ctypes.c_int, [D, P, P, P, ctypes.c_float, P, P]),
        "qgemm_workspace_bytes": (SZ, [D, I64]),
        "qgemm_w4a16": (ctypes.c_int, [D, P, P, I64, I64, P, P, P, I64, P, SZ, P]),
        "qgemm_w4a8": (ctypes.c_int, [D, P, P, I64, I64, P, P, P, P, I64, P, SZ, P]),
        "qgemm_quant_act_fp8": (ctypes.c_int, [P, I64, I64, I64, P, I64, P, P]),
        "qgemm_moe_grouped": (ctypes.c_int, [D, P, I32, I32, P, I64, I64, P, P, P, P, I64, P, SZ, P]),
        "qgemm_dequant_debug": (ctypes.c_int, [D, P, P, P]),
        "qgemm_device_status": (ctypes.c_int, [I32]),
        "qgemm_force_config": (ctypes.c_int, [I32, I32]),
        "qgemm_debug_stall": (ctypes.c_int, [I32, I32]),
        "qgemm_w4a16_noalloc": (ctypes.c_int, [D, P, P, I64, I64, P, P, I64, P]),
        "qgemm_plan": (ctypes.c_int, [D, I64, P]),
        "qgemm_moe_workspace_bytes": (SZ, [D, I32, I64]),
        "qgemm_moe_indexed_workspace_bytes": (SZ, [D, I32, I32, I64, I64]),
        "qgemm_act_copy_bytes": (SZ, [D, I64]),
        "qgemm_w4a4": (ctypes.c_int, [D, P, P, I64, I64, P, I64, P, P, P, I64, P, SZ, P]),
        "qgemm_quant_act_mxfp4": (ctypes.c_int, [P, I64, I64, I64, P, I64, P, I64, P]),
        "qgemm_host_staging_bytes": (SZ, [D, I64]),
        "qgemm_moe_indexed": (ctypes.c_int, [D, P, I32, I32, P, I64, I64, P, P, P, P, I64, P, I64, P, SZ, P]),
        "qgemm_w4a16_host": (ctypes.c_int, [D, P, P, I64, I64, P, P, P, I64, P, SZ, P, SZ, P]),
    }
    for name, (res, args) in sigs.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(status, what):
    if status != 0:
        raise QGemmError(status, what)


def _need(t, name, dtype, cuda=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def _row_major(t, name):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D tensor with unit column stride")


def check_desc(desc):
    d = desc.c()
    return lib().qgemm_check_desc(ctypes.byref(d))


def packed_bytes(desc):
    d = desc.c()
    n = lib().qgemm_packed_bytes(ctypes.byref(d))
    if n == 0:
        raise QGemmError(1, "packed_bytes")
    return int(n)


def repack(desc, codes, scales, zeros=None, out=None, num_experts=1, global_scale=None):
    """Canonical (codes uint8 [N, K/2], scales bf16-bits/E8M0/E4M3 [N, K/g], zeros) -> packed.

    For an MoE layer pass tensors with a leading expert dimension and num_experts=E.
    global_scale: NVFP4's per-tensor scale, a float or one per expert (default 1)."""
    nb = packed_bytes(desc)
    if out is None:
        out = torch.empty(nb * num_experts, dtype=torch.uint8, device=codes.device)
    L = lib()
    d = desc.c()
    for e in range(num_experts):
        c = codes[e] if num_experts > 1 else codes
        s = scales[e] if num_experts > 1 else scales
        z = None if zeros is None else (zeros[e] if num_experts > 1 else zeros)
        c, s = c.contiguous(), s.contiguous()
        z = None if z is None else z.contiguous()
        g = 1.0 if global_scale is None else global_scale
        g = float(g[e]) if isinstance(g, (list, tuple)) else float(g)
        _check(L.qgemm_repack_scaled(ctypes.byref(d), _ptr(c), _ptr(s), _ptr(z), g,
                                     ctypes.c_void_p(out.data_ptr() + e * nb), _stream()),
               "repack")
    return out


def workspace_bytes(desc, M_max):
    d = desc.c()
    return int(lib().qgemm_workspace_bytes(ctypes.byref(d), int(M_max)))


def workspace(desc, M_max, device="cuda"):
    """A zero-filled workspace for calls with M <= M_max (reusable across calls)."""
    n = workspace_bytes(desc, M_max)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def w4a16(desc, packed, X, chan_scale=None, out=None, ws=None, bias=None):
    """Y = X . dequant(W)^T (* chan_scale[n]) with BF16 X [M, K]."""
    _need(X, "X", torch.bfloat16)
    _row_major(X, "X")
    M = X.shape[0]
    if out is None:
        out = torch.empty(M, desc.N, dtype=torch.bfloat16, device=X.device)
    _need(out, "out", torch.bfloat16)
    _row_major(out, "out")
    if chan_scale is not None:
        _need(chan_scale, "chan_scale", torch.float32)
    if ws is None:
        ws = workspace(desc, M, X.device)
    d = desc.c()
    _check(lib().qgemm_w4a16(ctypes.byref(d), _ptr(packed), _ptr(X), M, X.stride(0),
                             _ptr(chan_scale), _ptr(bias), _ptr(out), out.stride(0), _ptr(ws),
                             ws.numel() * ws.element_size(), _stream()), "w4a16")
    return out


def quant_act_fp8(X, out=None, scale=None):
    """Tokenwise FP8 e4m3 quantization of BF16 X [M, K] -> (codes uint8 [M, K], s fp32 [M])."""
    _need(X, "X", torch.bfloat16)
    _row_major(X, "X")
    M, K = X.shape
    if out is None:
        out = torch.empty(M, K, dtype=torch.uint8, device=X.device)
    if scale is None:
        scale = torch.empty(M, dtype=torch.float32, device=X.device)
    _check(lib().qgemm_quant_act_fp8(_ptr(X), M, K, X.stride(0), _ptr(out), out.stride(0),
                                     _ptr(scale), _stream()), "quant_act_fp8")
    return out, scale


def w4a8(desc, packed, Xq, tok_scale, chan_scale=None, out=None, ws=None, bias=None):
    """Y = diag(tok_scale) . e4m3(Xq) . dequant(W)^T (* chan_scale[n])."""
    _need(Xq, "Xq", torch.uint8)
    _row_major(Xq, "Xq")
    _need(tok_scale, "tok_scale", torch.float32)
    M = Xq.shape[0]
    if out is None:
        out = torch.empty(M, desc.N, dtype=torch.bfloat16, device=Xq.device)
    if ws is None:
        ws = workspace(desc, M, Xq.device)
    d = desc.c()
    _check(lib().qgemm_w4a8(ctypes.byref(d), _ptr(packed), _ptr(Xq), M, Xq.stride(0),
                            _ptr(tok_scale), _ptr(chan_scale), _ptr(bias), _ptr(out), out.stride(0),
                            _ptr(ws),
                            ws.numel() * ws.element_size(), _stream()), "w4a8")
    return out


def quant_act_mxfp4(X, out=None, exps=None):
    """MXFP4 activations of BF16 X [M, K]: (codes uint8 [M, K/2], E8M0 exponents uint8
    [M, ceil(K/128)*4 rounded up to 16]) (see qgemm_quant_act_mxfp4)."""
    _row_major(X, "X")
    M, K = X.shape
    if out is None:
        out = torch.empty(M, K // 2, dtype=torch.uint8, device=X.device)
    if exps is None:
        exps = torch.empty(M, -(-((K // 32 + 3) // 4 * 4) // 16) * 16, dtype=torch.uint8,
                           device=X.device)
    _check(lib().qgemm_quant_act_mxfp4(_ptr(X), M, K, X.stride(0), _ptr(out), out.stride(0),
                                       _ptr(exps), exps.stride(0), _stream()), "quant_act_mxfp4")
    return out, exps


def w4a4(desc, packed, Xq, x_exps, chan_scale=None, out=None, ws=None, bias=None):
    """Dense W4A4: MXFP4 codes Xq [M, K/2] and exponents x_exps [M, >= ceil(K/128)*4] from
    quant_act_mxfp4, weights repacked with afmt "mxfp4"."""
    M = Xq.shape[0]
    if out is None:
        out = torch.empty(M, desc.N, dtype=torch.bfloat16, device=Xq.device)
    if ws is None:
        ws = workspace(desc, M, Xq.device)
    d = desc.c()
    _check(lib().qgemm_w4a4(ctypes.byref(d), _ptr(packed), _ptr(Xq), M, Xq.stride(0), _ptr(x_exps),
                            x_exps.stride(0), _ptr(chan_scale), _ptr(bias), _ptr(out),
                            out.stride(0), _ptr(ws), ws.numel() * ws.element_size(), _stream()),
           "w4a4")
    return out


def host_staging_bytes(desc, M_max):
    d = desc.c()
    return int(lib().qgemm_host_staging_bytes(ctypes.byref(d), int(M_max)))


def host_staging(desc, M_max, device="cuda"):
    """Device staging for w4a16_host calls with M <= M_max (reusable on one stream)."""
    return torch.empty(max(host_staging_bytes(desc, M_max), 256), dtype=torch.uint8, device=device)


def w4a16_host(desc, packed, X_host, out=None, staging=None, ws=None, chan_scale=None, bias=None):
    """Dense W4A16 with X [M, K] and Y [M, N] in host memory (BF16, pin them for speed):
    the copies in and out overlap the GEMM chunk by chunk.  Asynchronous on the current
    stream: synchronize before reading `out`."""
    _row_major(X_host, "X_host")
    if X_host.is_cuda:
        raise QGemmError("w4a16_host takes a host X; use w4a16 for device tensors")
    M = X_host.shape[0]
    if out is None:
        out = torch.empty(M, desc.N, dtype=torch.bfloat16, pin_memory=True)
    if staging is None:
        staging = host_staging(desc, M, device=packed.device)
    if ws is None:
        ws = workspace(desc, M, device=packed.device)
    d = desc.c()
    _check(lib().qgemm_w4a16_host(ctypes.byref(d), _ptr(packed), _ptr(X_host), M, X_host.stride(0),
                                  _ptr(chan_scale), _ptr(bias), _ptr(out), out.stride(0),
                                  _ptr(staging),
                                  staging.numel(), _ptr(ws), ws.numel(), _stream()), "w4a16_host")
    return out


def moe_workspace_bytes(desc, E, R):
    d = desc.c()
    return int(lib().qgemm_moe_workspace_bytes(ctypes.byref(d), int(E), int(R)))


def moe_workspace(desc, E, R, device="cuda"):
    """A zero-filled workspace that lets qgemm_moe_grouped use stream-K (reusable)."""
    return torch.zeros(max(moe_workspace_bytes(desc, E, R), 256), dtype=torch.uint8, device=device)


def moe_indexed_workspace_bytes(desc, E, T, R, fp8=False):
    d = desc.c()
    return int(lib().qgemm_moe_indexed_workspace_bytes(ctypes.byref(d), int(E),
                                                       AFMT["fp8" if fp8 else "bf16"], int(T), int(R)))


def moe_indexed_workspace(desc, E, T, R, fp8=False, device="cuda"):
    """A zero-filled workspace for qgemm_moe_indexed's fastest schedule (reusable)."""
    return torch.zeros(max(moe_indexed_workspace_bytes(desc, E, T, R, fp8), 256), dtype=torch.uint8,
                       device=device)


def act_copy_bytes(desc, x_rows):
    """Bytes of the FP16 activation copy (INT4 with BF16 scales; 0 for other formats)."""
    d = desc.c()
    return int(lib().qgemm_act_copy_bytes(ctypes.byref(d), int(x_rows)))


def _moe_min_ws(desc, x_rows, device):
    """The smallest workspace the MoE calls accept: the activation copy, or None."""
    n = act_copy_bytes(desc, x_rows)
    return None if n == 0 else torch.empty(n, dtype=torch.uint8, device=device)


def moe_grouped(desc, packed, E, X, offsets, tok_scale=None, out=None, ws=None, bias=None):
    """MoE grouped GEMM over expert-sorted rows X [R, K] (BF16, or uint8 e4m3 with
    tok_scale); offsets: int32 [E+1] on the device; ws: optional moe_workspace() (without
    one, whole tiles, and for INT4 with BF16 scales just the activation copy)."""
    fp8 = X.dtype == torch.uint8
    _need(offsets, "offsets", torch.int32)
    _row_major(X, "X")
    R = X.shape[0]
    if out is None:
        out = torch.empty(R, desc.N, dtype=torch.bfloat16, device=X.device)
    if ws is None:
        ws = _moe_min_ws(desc, R, X.device)
    d = desc.c()
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().qgemm_moe_grouped(ctypes.byref(d), _ptr(packed), E, AFMT["fp8" if fp8 else "bf16"],
                                   _ptr(X), R, X.stride(0), _ptr(tok_scale), _ptr(bias), _ptr(offsets),
                                   _ptr(out), out.stride(0), _ptr(ws), wsb, _stream()), "moe_grouped")
    return out


def moe_indexed(desc, packed, E, X, offsets, row_index, tok_scale=None, out=None, ws=None,
                bias=None):
    """MoE GEMM over rows gathered by index: X [T, K] in token order (BF16, or uint8 e4m3
    with tok_scale [T]); offsets int32 [E+1] and row_index int32 [R] on the device
    (row_index[r] < 0: padding).  Returns Y [R, N] in sorted order."""
    fp8 = X.dtype == torch.uint8
    _need(offsets, "offsets", torch.int32)
    _need(row_index, "row_index", torch.int32)
    _row_major(X, "X")
    R = row_index.numel()
    if out is None:
        out = torch.empty(R, desc.N, dtype=torch.bfloat16, device=X.device)
    if ws is None:
        ws = _moe_min_ws(desc, X.shape[0], X.device)
    d = desc.c()
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().qgemm_moe_indexed(ctypes.byref(d), _ptr(packed), E, AFMT["fp8" if fp8 else "bf16"],
                                   _ptr(X), X.shape[0], X.stride(0), _ptr(tok_scale), _ptr(bias),
                                   _ptr(offsets),
                                   _ptr(row_index), R, _ptr(out), out.stride(0), _ptr(ws), wsb,
                                   _stream()), "moe_indexed")
    return out


def dequant_debug(desc, packed):
    """BF16 W [N, K] decoded from the packed form by the GEMM's own register decoders."""
    out = torch.empty(desc.N, desc.K, dtype=torch.bfloat16, device=packed.device)
    d = desc.c()
    _check(lib().qgemm_dequant_debug(ctypes.byref(d), _ptr(packed), _ptr(out), _stream()),
           "dequant_debug")
    return out


def device_status(clear=True):
    """First device-side error since the last reset (0 = none); synchronizes."""
    return int(lib().qgemm_device_status(1 if clear else 0))


def force_config(token_tile=0, splits=0):
    """splits: >= 1 uniform K cut, -1 stream-K, 0 heuristic (see qgemm_force_config)."""
    _check(lib().qgemm_force_config(int(token_tile), int(splits)), "force_config")


def debug_stall(skip_first_x=0, timeout_ms=0):
    """Test aid for the bounded waits (see qgemm_debug_stall); (0, 0) restores the default."""
    _check(lib().qgemm_debug_stall(int(skip_first_x), int(timeout_ms)), "debug_stall")


def plan(desc, M):
    """The dense schedule for M rows: dict(token_tile, splits, sk_tiles, max_contrib, grid)."""
    out = (ctypes.c_int32 * 5)()
    d = desc.c()
    _check(lib().qgemm_plan(ctypes.byref(d), int(M), out), "plan")
    return dict(zip(("token_tile", "splits", "sk_tiles", "max_contrib", "grid"), list(out)))
