"""ctypes binding of the C ABI declared in ``include/fgemm.h``.

Argument marshalling only: every call goes straight to ``libfgemm.so`` and the
work runs in its CUDA kernels.  Matrices may be given as CUDA float32 torch
tensors (their ``data_ptr()`` is passed) or as raw device addresses (ints).
When no stream is given and a tensor is passed, torch's current stream on that
tensor's device is used; otherwise the legacy default stream (0).

There is no CPU fallback: if the library cannot be built or loaded, every call
raises.
"""

from __future__ import annotations

import ctypes
import threading

from . import _build

OP_N, OP_T = 0, 1
OK, ERR_INVALID_VALUE, ERR_LAUNCH, ERR_NOT_SUPPORTED, ERR_TIMEOUT = 0, 1, 2, 3, 4
MATH_FP32, MATH_TF32, MATH_3XTF32 = 0, 1, 2

_lock = threading.Lock()
_lib = None

_c_int, _c_float, _c_ll, _c_vp = ctypes.c_int, ctypes.c_float, ctypes.c_longlong, ctypes.c_void_p


class FgemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, status_string(status)))


def library() -> ctypes.CDLL:
    """Load (building first if the sources are newer) ``libfgemm.so``."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            lib = ctypes.CDLL(path)
            sig = {
                "fgemm_sgemm": [_c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _c_vp, _c_int,
                                _c_vp, _c_int, _c_float, _c_vp, _c_int, _c_vp],
                "fgemm_sgemm_bias_relu": [_c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _c_vp,
                                          _c_int, _c_vp, _c_int, _c_float, _c_vp, _c_int, _c_vp,
                                          _c_int, _c_vp],
                "fgemm_sgemm_row_bias_relu": [_c_int, _c_int, _c_int, _c_int, _c_int, _c_float,
                                              _c_vp, _c_int, _c_vp, _c_int, _c_float, _c_vp,
                                              _c_int, _c_vp, _c_int, _c_vp],
                "fgemm_sgemm_strided_batched": [_c_int, _c_int, _c_int, _c_int, _c_int, _c_float,
                                                _c_vp, _c_int, _c_ll, _c_vp, _c_int, _c_ll,
                                                _c_float, _c_vp, _c_int, _c_ll, _c_int, _c_vp],
                "fgemm_gemm_explicit": [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float,
                                        _c_vp, _c_int, _c_ll, _c_vp, _c_int, _c_ll, _c_float,
                                        _c_vp, _c_int, _c_ll, _c_int, _c_vp, _c_int, _c_vp],
                "fgemm_gemm_math": [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float,
                                    _c_vp, _c_int, _c_ll, _c_vp, _c_int, _c_ll, _c_float,
                                    _c_vp, _c_int, _c_ll, _c_int, _c_vp, _c_int, _c_vp],
                "fgemm_device_status": [_c_int],
                "fgemm_select_config": [_c_int] * 8,
                "fgemm_launch_count": [_c_int] * 9,
                "fgemm_num_configs": [],
                "fgemm_config_name": [_c_int],
                "fgemm_status_string": [_c_int],
            }
            for name, argtypes in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = argtypes
                fn.restype = _c_int
            lib.fgemm_sgemm_splitk.argtypes = [_c_int, _c_int, _c_int, _c_int, _c_int, _c_float,
                                               _c_vp, _c_int, _c_vp, _c_int, _c_float, _c_vp,
                                               _c_int, _c_vp, _c_int, _c_int, _c_vp,
                                               ctypes.c_size_t, _c_vp]
            lib.fgemm_sgemm_splitk.restype = _c_int
            lib.fgemm_sgemm_splitk_noalloc.argtypes = [_c_int, _c_int, _c_int, _c_int, _c_int,
                                                       _c_float, _c_vp, _c_int, _c_vp, _c_int,
                                                       _c_float, _c_vp, _c_int, _c_vp, _c_int,
                                                       _c_int, _c_vp]
            lib.fgemm_sgemm_splitk_noalloc.restype = _c_int
            lib.fgemm_splitk_workspace_size.argtypes = [_c_int, _c_int, _c_int, _c_int]
            lib.fgemm_splitk_workspace_size.restype = ctypes.c_size_t
            lib.fgemm_staged_workspace_size.argtypes = [_c_int] * 6
            lib.fgemm_staged_workspace_size.restype = ctypes.c_size_t
            lib.fgemm_staged_choice.argtypes = [_c_int] * 10 + [ctypes.c_size_t, _c_int]
            lib.fgemm_staged_choice.restype = _c_int
            lib.fgemm_sgemm_staged.argtypes = [_c_int, _c_int, _c_int, _c_int, _c_int, _c_float,
                                               _c_vp, _c_int, _c_ll, _c_vp, _c_int, _c_ll,
                                               _c_float, _c_vp, _c_int, _c_ll, _c_int, _c_vp,
                                               _c_int, _c_int, _c_vp, ctypes.c_size_t, _c_vp]
            lib.fgemm_sgemm_staged.restype = _c_int
            lib.fgemm_math_staged_workspace_size.argtypes = [_c_int] * 7
            lib.fgemm_math_staged_workspace_size.restype = ctypes.c_size_t
            lib.fgemm_math_staged_choice.argtypes = [_c_int] * 11 + [ctypes.c_size_t, _c_int]
            lib.fgemm_math_staged_choice.restype = _c_int
            lib.fgemm_gemm_math_staged.argtypes = [_c_int] + lib.fgemm_sgemm_staged.argtypes
            lib.fgemm_gemm_math_staged.restype = _c_int
            lib.fgemm_math_supported.argtypes = [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                                 _c_float, _c_vp, _c_int, _c_ll, _c_vp, _c_int,
                                                 _c_ll, _c_int]
            lib.fgemm_math_supported.restype = _c_int
            lib.fgemm_debug_withhold_tensor_core.argtypes = [_c_int, _c_ll]
            lib.fgemm_debug_withhold_tensor_core.restype = None
            lib.fgemm_config_name.restype = ctypes.c_char_p
            lib.fgemm_status_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    if hasattr(x, "data_ptr"):
        if x.numel() and (not x.is_cuda or x.dtype.itemsize != 4 or not x.is_floating_point()):
            raise TypeError("fgemm takes CUDA float32 tensors (got %s on %s)" % (x.dtype, x.device))
        return x.data_ptr() or None
    raise TypeError("expected a CUDA tensor or a device address, got %r" % type(x))


def _stream(stream, *tensors):
    if stream is None:
        for t in tensors:
            if hasattr(t, "is_cuda") and t.is_cuda:
                import torch
                return torch.cuda.current_stream(t.device).cuda_stream
        return None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream  # a torch.cuda.Stream


def _check(status: int, where: str):
    if status != OK:
        raise FgemmError(status, where)


def status_string(status: int) -> str:
    return library().fgemm_status_string(int(status)).decode()


def num_configs() -> int:
    return library().fgemm_num_configs()


def config_name(config: int):
    name = library().fgemm_config_name(int(config))
    return name.decode() if name else None


def select_config(transa, transb, M, N, K, batch, aligned, num_sms) -> int:
    return library().fgemm_select_config(int(transa), int(transb), M, N, K, batch,
                                         1 if aligned else 0, num_sms)


def launch_count(config, transa, transb, M, N, K, batch, aligned, num_sms) -> int:
    """``fgemm_launch_count``: kernel launches of one call (config < 0: as selected)."""
    return library().fgemm_launch_count(int(config), int(transa), int(transb), M, N, K, batch,
                                        1 if aligned else 0, num_sms)


def sgemm(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None,
          check=True) -> int:
    """``fgemm_sgemm``: C = alpha*op(A)*op(B) + beta*C (row-major, see include/fgemm.h)."""
    st = library().fgemm_sgemm(int(transa), int(transb), M, N, K, alpha, _ptr(A), lda, _ptr(B),
                               ldb, beta, _ptr(C), ldc, _stream(stream, C, A, B))
    if check:
        _check(st, "fgemm_sgemm")
    return st


def sgemm_bias_relu(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias,
                    apply_relu, stream=None, check=True) -> int:
    """``fgemm_sgemm_bias_relu``: C = relu?(alpha*op(A)*op(B) + beta*C + bias[col])."""
    st = library().fgemm_sgemm_bias_relu(int(transa), int(transb), M, N, K, alpha, _ptr(A), lda,
                                         _ptr(B), ldb, beta, _ptr(C), ldc, _ptr(bias),
                                         1 if apply_relu else 0, _stream(stream, C, A, B))
    if check:
        _check(st, "fgemm_sgemm_bias_relu")
    return st


def sgemm_row_bias_relu(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, row_bias,
                        apply_relu, stream=None, check=True) -> int:
    """``fgemm_sgemm_row_bias_relu``: C = relu?(alpha*op(A)*op(B) + beta*C + row_bias[row])."""
    st = library().fgemm_sgemm_row_bias_relu(int(transa), int(transb), M, N, K, alpha, _ptr(A),
                                             lda, _ptr(B), ldb, beta, _ptr(C), ldc, _ptr(row_bias),
                                             1 if apply_relu else 0, _stream(stream, C, A, B))
    if check:
        _check(st, "fgemm_sgemm_row_bias_relu")
    return st


def sgemm_strided_batched(transa, transb, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta,
                          C, ldc, strideC, batch, stream=None, check=True) -> int:
    """``fgemm_sgemm_strided_batched``: the plain GEMM on batch offsets b*stride."""
    st = library().fgemm_sgemm_strided_batched(
        int(transa), int(transb), M, N, K, alpha, _ptr(A), lda, strideA, _ptr(B), ldb, strideB,
        beta, _ptr(C), ldc, strideC, batch, _stream(stream, C, A, B))
    if check:
        _check(st, "fgemm_sgemm_strided_batched")
    return st


def gemm_explicit(config, transa, transb, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta,
                  C, ldc, strideC, batch, bias=None, apply_relu=False, stream=None,
                  check=True) -> int:
    """``fgemm_gemm_explicit``: every option, with an explicit kernel configuration."""
    st = library().fgemm_gemm_explicit(
        int(config), int(transa), int(transb), M, N, K, alpha, _ptr(A), lda, strideA, _ptr(B), ldb,
        strideB, beta, _ptr(C), ldc, strideC, batch, _ptr(bias), 1 if apply_relu else 0,
        _stream(stream, C, A, B))
    if check:
        _check(st, "fgemm_gemm_explicit")
    return st


def gemm_math(math, transa, transb, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C,
              ldc, strideC, batch, bias=None, apply_relu=False, stream=None, check=True) -> int:
    """``fgemm_gemm_math``: FP32 CUDA cores (MATH_FP32) or tcgen05 TF32 / 3xTF32."""
    st = library().fgemm_gemm_math(
        int(math), int(transa), int(transb), M, N, K, alpha, _ptr(A), lda, strideA, _ptr(B), ldb,
        strideB, beta, _ptr(C), ldc, strideC, batch, _ptr(bias), 1 if apply_relu else 0,
        _stream(stream, C, A, B))
    if check:
        _check(st, "fgemm_gemm_math")
    return st


def math_supported(math, transa, transb, M, N, K, alpha, A, lda, strideA, B, ldb, strideB,
                   batch) -> int:
    """``fgemm_math_supported``: 1 if ``gemm_math`` runs the requested arithmetic for these
    operands, 0 if it would use the FP32 CUDA-core kernel instead, -1 for a bad ``math``.
    Host-only; the pointers are only tested for alignment."""
    return library().fgemm_math_supported(int(math), int(transa), int(transb), M, N, K, alpha,
                                          _ptr(A), lda, strideA, _ptr(B), ldb, strideB, batch)


def device_status(clear=True) -> int:
    """``fgemm_device_status``: ERR_TIMEOUT if a tensor-core wait ran out (call after a sync)."""
    return library().fgemm_device_status(1 if clear else 0)


def debug_withhold_tensor_core(k_block: int, wait_limit_ns: int = 0) -> None:
    """Testing: ``fgemm_debug_withhold_tensor_core`` (k_block < 0 restores normal runs)."""
    library().fgemm_debug_withhold_tensor_core(int(k_block), int(wait_limit_ns))


def splitk_workspace_size(M, N, K, splits) -> int:
    """``fgemm_splitk_workspace_size``: bytes of workspace fgemm_sgemm_splitk needs (0: invalid)."""
    return int(library().fgemm_splitk_workspace_size(M, N, K, splits))


def sgemm_splitk(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias, apply_relu,
                 splits, workspace, workspace_bytes, stream=None, check=True) -> int:
    """``fgemm_sgemm_splitk``: split-K GEMM with a caller-owned workspace."""
    st = library().fgemm_sgemm_splitk(
        int(transa), int(transb), M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C), ldc,
        _ptr(bias), 1 if apply_relu else 0, int(splits), _ptr(workspace), int(workspace_bytes),
        _stream(stream, C, A, B))
    if check:
        _check(st, "fgemm_sgemm_splitk")
    return st


# FGEMM_MAX_DIM of include/fgemm.h: the largest M, N or K a call takes (2^31 - 256);
# larger sizes return FGEMM_ERR_NOT_SUPPORTED.
MAX_DIM = 2**31 - 256


# FGEMM_NOALLOC_SCRATCH_BYTES of include/fgemm.h: the fixed scratch array behind
# fgemm_sgemm_splitk_noalloc.
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


def sgemm_splitk_noalloc(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias,
                         apply_relu, splits, stream=None, check=True) -> int:
    """``fgemm_sgemm_splitk_noalloc``: split-K GEMM whose partial products live in the
    library's fixed device array instead of a caller workspace (for callers that may
    not allocate device memory)."""
    st = library().fgemm_sgemm_splitk_noalloc(
        int(transa), int(transb), M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C), ldc,
        _ptr(bias), 1 if apply_relu else 0, int(splits), _stream(stream, C, A, B))
    if check:
        _check(st, "fgemm_sgemm_splitk_noalloc")
    return st


# stage = -1 for fgemm_sgemm_staged: the launch-time model chooses.
STAGE_AUTO = -1


def staged_workspace_size(transa, transb, M, N, K, batch) -> int:
    """``fgemm_staged_workspace_size``: bytes of workspace fgemm_sgemm_staged needs."""
    return int(library().fgemm_staged_workspace_size(int(transa), int(transb), M, N, K, batch))


def staged_choice(transa, transb, M, N, K, batch, shared_a, shared_b, aligned_a, aligned_b,
                  num_sms, workspace_bytes=None) -> int:
    """``fgemm_staged_choice``: which operands a staged call copies into its workspace
    (bit 0: A, bit 1: B) by the launch-time model; host-only.  workspace_bytes=None:
    the full fgemm_staged_workspace_size."""
    if workspace_bytes is None:
        workspace_bytes = staged_workspace_size(transa, transb, M, N, K, max(1, batch))
    return library().fgemm_staged_choice(int(transa), int(transb), M, N, K, batch,
                                         1 if shared_a else 0, 1 if shared_b else 0,
                                         1 if aligned_a else 0, 1 if aligned_b else 0,
                                         int(workspace_bytes), num_sms)


def sgemm_staged(transa, transb, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc,
                 strideC, batch, bias, apply_relu, stage, workspace, workspace_bytes,
                 stream=None, check=True) -> int:
    """``fgemm_sgemm_staged``: the GEMM after copying operands into a caller workspace
    (transposed k-major, or re-pitched when unaligned; stage = STAGE_AUTO: the copies the
    model finds faster among those that fit)."""
    st = library().fgemm_sgemm_staged(
        int(transa), int(transb), M, N, K, alpha, _ptr(A), lda, strideA, _ptr(B), ldb, strideB,
        beta, _ptr(C), ldc, strideC, batch, _ptr(bias), 1 if apply_relu else 0, int(stage),
        _ptr(workspace), int(workspace_bytes), _stream(stream, C, A, B))
    if check:
        _check(st, "fgemm_sgemm_staged")
    return st


def math_staged_workspace_size(math, transa, transb, M, N, K, batch) -> int:
    """``fgemm_math_staged_workspace_size``: bytes of workspace fgemm_gemm_math_staged needs
    for both copies."""
    return int(library().fgemm_math_staged_workspace_size(int(math), int(transa), int(transb), M,
                                                          N, K, batch))


def math_staged_choice(math, transa, transb, M, N, K, batch, shared_a, shared_b, aligned_a,
                       aligned_b, num_sms, workspace_bytes=None) -> int:
    """``fgemm_math_staged_choice``: the copies fgemm_gemm_math_staged makes with
    stage = STAGE_AUTO (bit 0: A, bit 1: B); host-only.  workspace_bytes=None: the full
    fgemm_math_staged_workspace_size."""
    if workspace_bytes is None:
        workspace_bytes = math_staged_workspace_size(math, transa, transb, M, N, K, max(1, batch))
    return library().fgemm_math_staged_choice(int(math), int(transa), int(transb), M, N, K, batch,
                                              1 if shared_a else 0, 1 if shared_b else 0,
                                              1 if aligned_a else 0, 1 if aligned_b else 0,
                                              int(workspace_bytes), num_sms)


def gemm_math_staged(math, transa, transb, M, N, K, alpha, A, lda, strideA, B, ldb, strideB,
                     beta, C, ldc, strideC, batch, bias, apply_relu, stage, workspace,
                     workspace_bytes, stream=None, check=True) -> int:
    """``fgemm_gemm_math_staged``: fgemm_gemm_math after copying operands K-major into a
    caller workspace (stage = STAGE_AUTO: the library's choice among the copies that fit)."""
    st = library().fgemm_gemm_math_staged(
        int(math), int(transa), int(transb), M, N, K, alpha, _ptr(A), lda, strideA, _ptr(B), ldb,
        strideB, beta, _ptr(C), ldc, strideC, batch, _ptr(bias), 1 if apply_relu else 0,
        int(stage), _ptr(workspace), int(workspace_bytes), _stream(stream, C, A, B))
    if check:
        _check(st, "fgemm_gemm_math_staged")
    return st
