"""FP64 CPU oracle for the row-major FP32 GEMM family (test infrastructure).

This package is the checker, not the product.  Only ``tests/``, the smoke check
in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.
The CUDA library never calls it and shares no code with it.

What it computes is the plain definition (see ``oracle.c`` for the citations):

    C[i][j] = relu?( alpha * sum_k op(A)[i][k] * op(B)[k][j] + beta * C0[i][j] + bias[j]
                     + row_bias[i] )

evaluated in double, one element at a time, with the k-sum in ascending order.
Each call also returns ``mag[i][j] = |alpha| sum_k |op(A)[i][k]| |op(B)[k][j]|
+ |beta| |C0[i][j]| + |bias[j]| + |row_bias[i]|``, the scale of the per-element bound used by
the tests (the bound itself lives in the tests).

The C source is compiled with gcc on first use (``build()``) into a shared
object beside it; nothing here needs CUDA.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_default = None

_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)

CFLAGS = ["-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
          "-Wall", "-Wextra"]


def compile_source(src: str, out: str) -> str:
    """Compile one oracle C file into a shared object with the oracle's flags."""
    tmp = out + ".tmp.%d" % os.getpid()
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` if it is missing or stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_source(SOURCE, _LIB)
    return _LIB


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _fptr(a):
    if a is None:
        return None
    if not (isinstance(a, np.ndarray) and a.dtype == np.float32 and a.flags.c_contiguous):
        raise TypeError("oracle inputs must be C-contiguous float32 numpy arrays")
    return a.ctypes.data_as(_f32p)


def _as_f32(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # a CPU torch tensor
        a = a.detach().cpu().contiguous().numpy()
    return np.ascontiguousarray(a, dtype=np.float32)


class Oracle:
    """ctypes view of one compiled oracle shared object."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.oracle_gemm.restype = ctypes.c_int
        lib.oracle_gemm.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_float, _f32p, ctypes.c_int64, _f32p, ctypes.c_int64, ctypes.c_float,
            _f32p, ctypes.c_int64, _f32p, _f32p, ctypes.c_int, _i64p, ctypes.c_int64,
            _f64p, _f64p, ctypes.c_int]
        lib.oracle_gemm_strided_batched.restype = ctypes.c_int
        lib.oracle_gemm_strided_batched.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_float, _f32p, ctypes.c_int64, ctypes.c_int64, _f32p, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_float, _f32p, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, _f64p, _f64p, ctypes.c_int]
        self.path = path
        self._lib = lib

    def gemm(self, ta, tb, M, N, K, alpha, A, lda, B, ldb, beta=0.0, C0=None, ldc=None,
             bias=None, relu=False, rows=None, threads=None, want_mag=True, row_bias=None):
        """FP64 reference of one (possibly fused) row-major GEMM.

        ``A``, ``B``, ``C0`` are the flat float32 storage the leading dimensions
        index into; ``ta``/``tb`` are 0 (no transpose) or 1 (transpose).  ``bias``
        has one value per column (length N), ``row_bias`` one per row (length M).
        Returns ``(out, mag)`` as float64 arrays of shape ``(len(rows) or M, N)``
        (``mag`` is None when ``want_mag`` is false).
        """
        A, B, C0, bias = _as_f32(A), _as_f32(B), _as_f32(C0), _as_f32(bias)
        row_bias = _as_f32(row_bias)
        ldc = N if ldc is None else ldc
        if rows is None:
            nrows, rows_arr, rptr = M, None, None
        else:
            rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
            nrows, rptr = rows_arr.size, rows_arr.ctypes.data_as(_i64p)
        out = np.zeros((nrows, N), dtype=np.float64)
        mag = np.zeros((nrows, N), dtype=np.float64) if want_mag else None
        rc = self._lib.oracle_gemm(
            int(ta), int(tb), M, N, K, float(alpha), _fptr(A), lda, _fptr(B), ldb, float(beta),
            _fptr(C0), ldc, _fptr(bias), _fptr(row_bias), 1 if relu else 0, rptr, nrows,
            out.ctypes.data_as(_f64p), mag.ctypes.data_as(_f64p) if mag is not None else None,
            int(threads or default_threads()))
        if rc != 0:
            raise ValueError("oracle_gemm rejected its arguments (code %d)" % rc)
        return out, mag

    def gemm_strided_batched(self, ta, tb, M, N, K, alpha, A, lda, strideA, B, ldb, strideB,
                             beta, C0, ldc, strideC, batch, threads=None, want_mag=True):
        """FP64 reference of a strided batch; returns arrays of shape (batch, M, N)."""
        A, B, C0 = _as_f32(A), _as_f32(B), _as_f32(C0)
        out = np.zeros((batch, M, N), dtype=np.float64)
        mag = np.zeros((batch, M, N), dtype=np.float64) if want_mag else None
        rc = self._lib.oracle_gemm_strided_batched(
            int(ta), int(tb), M, N, K, float(alpha), _fptr(A), lda, strideA, _fptr(B), ldb,
            strideB, float(beta), _fptr(C0), ldc, strideC, batch, out.ctypes.data_as(_f64p),
            mag.ctypes.data_as(_f64p) if mag is not None else None,
            int(threads or default_threads()))
        if rc != 0:
            raise ValueError("oracle_gemm_strided_batched rejected its arguments (code %d)" % rc)
        return out, mag


def default() -> Oracle:
    """The oracle built from ``oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def gemm(*args, **kwargs):
    return default().gemm(*args, **kwargs)


def gemm_strided_batched(*args, **kwargs):
    return default().gemm_strided_batched(*args, **kwargs)
