"""W4A16 (bf16 activation x INT4 weight, group-128) linear layer for GB300.

The compute lives in the CUDA library ``libw4a16.so`` (C ABI declared in
``include/w4a16.h``); the functions below are its Python binding, with the
same names.  The library is loaded on first use and a missing build raises.
"""
from ._lib import (  # noqa: F401
    EPI_BIAS, EPI_NONE, EPI_SILU_MUL, GROUP, PATH_AUTO, PATH_NAMES, PATH_SKINNY, PATH_TCGEN05,
    W4A16Error, load, w4a16_debug_forced_timeout, w4a16_dequant_ref, w4a16_device_status,
    w4a16_dequant_ref_f16, w4a16_gemm, w4a16_gemm_f16, w4a16_gemm_fused, w4a16_gemm_grouped,
    w4a16_grouped_workspace_bytes,
    w4a16_describe_plan, w4a16_kernel_name, w4a16_pack, w4a16_packed_check,
    w4a16_packed_bytes, w4a16_quantize_rtn, w4a16_select_path, w4a16_workspace_bytes,
    w8a8_fp8_gemm, w8a8_fp8_pack_weight, w8a8_fp8_packed_bytes, w8a8_fp8_quantize_act,
    w8a8_fp8_quantize_weight, w8a8_fp8_workspace_bytes)
