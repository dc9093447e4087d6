"""fgemm: single-GPU FP32 GEMM for NVIDIA GB300 (sm_103a), hand-written CUDA kernels.

The product is the C-ABI shared library ``libfgemm.so`` (declared in
``include/fgemm.h``).  This package is its thin Python binding: the functions
below marshal arguments and call the library; all work runs in its kernels.
"""

from ._binding import (  # noqa: F401
    ERR_INVALID_VALUE,
    ERR_LAUNCH,
    ERR_NOT_SUPPORTED,
    ERR_TIMEOUT,
    MATH_3XTF32,
    MATH_FP32,
    MATH_TF32,
    OK,
    OP_N,
    OP_T,
    FgemmError,
    config_name,
    debug_withhold_tensor_core,
    device_status,
    gemm_math,
    gemm_math_staged,
    gemm_explicit,
    launch_count,
    library,
    math_staged_choice,
    math_staged_workspace_size,
    math_supported,
    num_configs,
    select_config,
    sgemm,
    sgemm_bias_relu,
    sgemm_row_bias_relu,
    MAX_DIM,
    NOALLOC_SCRATCH_BYTES,
    STAGE_AUTO,
    sgemm_splitk,
    sgemm_splitk_noalloc,
    sgemm_staged,
    staged_choice,
    staged_workspace_size,
    splitk_workspace_size,
    sgemm_strided_batched,
    status_string,
)
