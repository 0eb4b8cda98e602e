"""CPU oracle of the quantized-weight GEMM (float64, numpy).

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the CPU legs of
bench.py, never by the product package.  See qgemm_oracle.py for what it computes.
"""
from . import formats
from .qgemm_oracle import (WFMTS, unpack_nibbles, scale_values, dequant, dequant_bf16, gemm,
                           w4a16, quant_act_fp8, w4a8, moe_grouped, moe_indexed, tolerance_ok,
                           quant_act_mxfp4, dequant_act_mxfp4, w4a4)

__all__ = ["formats", "WFMTS", "unpack_nibbles", "scale_values", "dequant", "dequant_bf16",
           "gemm", "w4a16", "quant_act_fp8", "w4a8", "moe_grouped", "moe_indexed",
           "tolerance_ok", "quant_act_mxfp4", "dequant_act_mxfp4", "w4a4"]
