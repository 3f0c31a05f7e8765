"""GB300 (sm_103a) dense GEMM: C = A . B with bf16/fp16, block-scaled (MX family) or NVFP4
operands, fp32 accumulation.

The compute runs in the CUDA library ``libdtc_gemm.so`` (C ABI in ``include/dtc_gemm.h``). This
package is a thin ctypes binding with the same function names: it checks and marshals torch
tensors (device pointers, sizes, the current stream) and raises ``GemmError`` on a non-OK status.
There is no CPU fallback: if the library is missing, every call raises.
"""
from ._binding import (  # noqa: F401
    GEMM_LAYOUT_NN,
    GEMM_LAYOUT_NT,
    GEMM_LAYOUT_TN,
    GEMM_LAYOUT_TT,
    GEMM_VARIANT_1CTA,
    GEMM_VARIANT_2CTA,
    GEMM_VARIANT_AUTO,
    GEMM_VARIANT_SPLITK,
    GB300_MODEL,
    GemmError,
    gemm_bf16,
    gemm_device_model_query,
    gemm_ex,
    gemm_ex_static_workspace,
    gemm_f16,
    gemm_last_error,
    gemm_mxfp8,
    gemm_nvfp4,
    gemm_nvfp4_workspace_size,
    gemm_plan,
    gemm_sp,
    gemm_sp_workspace_size,
    gemm_stream_status,
    gemm_workspace_size,
    lib,
    library_path,
)
