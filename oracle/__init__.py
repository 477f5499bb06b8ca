"""The oracle: a slow, plain CPU statement of C = alpha*op(A)*op(B) + beta*C.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the bench's CPU
baseline import this package; the GPU library never does, and the two share no
code.  The arithmetic lives in oracle_gemm.c (double accumulation in strict
increasing k, exact products); this module only marshals numpy arrays into it.

Citations for the definition are in oracle_gemm.c's header: the full-SGEMM
sidenote of "Optimizing GEMM on Apple's M5 from scratch, Part 1" (Introduction)
and its naive three-loop kernel, the ijk/ikj loops of "From a C loop to a GPU
kernel" ("The first loop"), and the nn/tn/nt variant table of "Metal GEMM
Kernels for LoRA Training on Apple Silicon" (section 2).
"""
import ctypes
import os

import numpy as np

from . import build_oracle

F32 = 0
F16 = 1
BF16 = 2
FORMATS = {"f32": F32, "f16": F16, "bf16": BF16}

_lib = None


def bind(path: str):
    """ctypes handle on an oracle shared object at `path` (the tests also bind
    deliberately broken builds of the same source to show the pins catch them)."""
    lib = ctypes.CDLL(path)
    i64, dbl, vp, ci = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
    lib.oracle_gemm.argtypes = [ci, ci, i64, i64, i64, ci, dbl, dbl, vp, i64, vp, i64, vp,
                                i64, vp, vp, ci]
    lib.oracle_gemm.restype = ci
    lib.oracle_gemm_points.argtypes = [ci, ci, i64, i64, i64, ci, dbl, dbl, vp, i64, vp, i64,
                                       vp, i64, vp, vp, i64, vp, vp, ci]
    lib.oracle_gemm_points.restype = ci
    lib.oracle_bias_act.argtypes = [vp, i64, i64, i64, vp, ci]
    lib.oracle_bias_act.restype = ci
    lib.oracle_gelu.argtypes = [dbl]
    lib.oracle_gelu.restype = dbl
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_double.restype = dbl
    lib.oracle_double_to_half_rne.argtypes = [dbl]
    lib.oracle_double_to_half_rne.restype = ctypes.c_uint16
    lib.oracle_half_array_to_double.argtypes = [vp, vp, i64]
    lib.oracle_half_array_to_double.restype = None
    lib.oracle_double_array_to_half_rne.argtypes = [vp, vp, i64]
    lib.oracle_double_array_to_half_rne.restype = None
    lib.oracle_bf16_array_to_double.argtypes = [vp, vp, i64]
    lib.oracle_bf16_array_to_double.restype = None
    lib.oracle_double_array_to_bf16_rne.argtypes = [vp, vp, i64]
    lib.oracle_double_array_to_bf16_rne.restype = None
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = bind(build_oracle.build())
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _dtype_code(a: np.ndarray, fmt=None) -> int:
    """Element format of an operand array.  bfloat16 has no numpy dtype: pass
    its bit patterns as uint16 with fmt='bf16'."""
    if fmt is not None:
        return FORMATS[fmt]
    if a.dtype == np.float32:
        return F32
    if a.dtype in (np.float16, np.uint16):
        return F16
    raise TypeError(f"oracle takes float32, float16 or (fmt='bf16') uint16 arrays, got {a.dtype}")


def _ld(a: np.ndarray) -> int:
    """Leading dimension (elements) of a 2-D row-major array view."""
    if a.ndim != 2:
        raise ValueError("operands are 2-D")
    if a.size == 0:
        return max(a.shape[1], 1)
    if a.shape[1] > 1 and a.strides[1] != a.itemsize:
        raise ValueError("rows must be contiguous")
    return a.strides[0] // a.itemsize if a.shape[0] > 1 else max(a.shape[1], 1)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _shape(transA, transB, A, B):
    M, K = (A.shape[1], A.shape[0]) if transA else (A.shape[0], A.shape[1])
    Kb, N = (B.shape[1], B.shape[0]) if transB else (B.shape[0], B.shape[1])
    if K != Kb:
        raise ValueError(f"inner dimensions differ: {K} vs {Kb}")
    return M, N, K


def gemm_ref(A, B, C=None, transA=False, transB=False, alpha=1.0, beta=0.0, threads=None,
             lib=None, fmt=None):
    """(ref, mag) for C_out = alpha*op(A)@op(B) + beta*C, both float64 [M, N].

    A, B, C are numpy float32 or float16 arrays (2-D row-major views; an ld
    larger than the row is taken from the strides).  op(X) = X.T when the
    trans flag is set, i.e. a transposed operand is stored [K, M] / [N, K].
    C is read only when beta != 0.
    """
    dt = _dtype_code(A, fmt)
    if _dtype_code(B, fmt) != dt or (C is not None and _dtype_code(C, fmt) != dt):
        raise TypeError("A, B and C must have one dtype")
    M, N, K = _shape(transA, transB, A, B)
    ref = np.empty((M, N), dtype=np.float64)
    mag = np.empty((M, N), dtype=np.float64)
    if beta != 0.0 and C is None:
        raise ValueError("beta != 0 needs C")
    ldc = _ld(C) if (C is not None and beta != 0.0) else max(N, 1)
    rc = (lib or _load()).oracle_gemm(int(transA), int(transB), M, N, K, dt, float(alpha),
                                      float(beta), _ptr(A), _ld(A), _ptr(B), _ld(B),
                                      _ptr(C) if beta != 0.0 else None, ldc,
                                      ref.ctypes.data, mag.ctypes.data,
                                      threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_gemm failed with code {rc}")
    return ref, mag


def gemm_ref_points(A, B, rows, cols, C=None, transA=False, transB=False, alpha=1.0, beta=0.0,
                    threads=None, fmt=None):
    """(ref, mag) at the output positions (rows[p], cols[p]); float64 [npts]."""
    dt = _dtype_code(A, fmt)
    M, N, K = _shape(transA, transB, A, B)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("rows and cols differ in length")
    ref = np.empty(rows.shape, dtype=np.float64)
    mag = np.empty(rows.shape, dtype=np.float64)
    if beta != 0.0 and C is None:
        raise ValueError("beta != 0 needs C")
    ldc = _ld(C) if (C is not None and beta != 0.0) else max(N, 1)
    rc = _load().oracle_gemm_points(int(transA), int(transB), M, N, K, dt, float(alpha),
                                    float(beta), _ptr(A), _ld(A), _ptr(B), _ld(B),
                                    _ptr(C) if beta != 0.0 else None, ldc,
                                    rows.ctypes.data, cols.ctypes.data, rows.size,
                                    ref.ctypes.data, mag.ctypes.data,
                                    threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_points failed with code {rc}")
    return ref, mag


ACTS = {"none": 0, "relu": 1, "gelu": 2}


def bias_act(x, bias=None, act="none", cols_index=None):
    """act(x + bias[j]) elementwise in double ("From a C loop to a GPU kernel",
    section "Fusion": per-output bias, then the activation).  x: float64 [M, N]
    (or [npts] with cols_index giving each point's column); bias: None or a
    length-N array of any oracle dtype (bfloat16 as uint16 with fmt handled by
    the caller: pass float64 values); act: 'none', 'relu' or 'gelu' (exact,
    v * Phi(v)).  Returns a new float64 array."""
    x = np.array(x, dtype=np.float64, copy=True)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float64)
    if x.ndim == 1:
        # points: one row whose k-th entry takes the bias of its own column
        if b is not None:
            b = np.ascontiguousarray(b[np.asarray(cols_index, dtype=np.int64)])
        x2 = x.reshape(1, -1)
    else:
        x2 = x
    rows, cols = x2.shape
    rc = _load().oracle_bias_act(x2.ctypes.data, rows, cols, cols,
                                 None if b is None else b.ctypes.data, ACTS[act])
    if rc != 0:
        raise RuntimeError("oracle_bias_act failed")
    return x2.reshape(x.shape)


def gelu(v):
    """The oracle's exact gelu, elementwise (float64)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    f = _load().oracle_gelu
    return np.vectorize(lambda t: f(float(t)))(v)


def half_to_double(h) -> np.ndarray:
    """binary16 bit patterns (uint16 or float16 array) -> float64, exact."""
    h = np.ascontiguousarray(h).view(np.uint16)
    out = np.empty(h.shape, dtype=np.float64)
    _load().oracle_half_array_to_double(h.ctypes.data, out.ctypes.data, h.size)
    return out


def round_half_rne(x) -> np.ndarray:
    """float64 -> binary16 bit patterns (uint16), round to nearest, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_double_array_to_half_rne(x.ctypes.data, out.ctypes.data, x.size)
    return out


def bf16_to_double(h) -> np.ndarray:
    """bfloat16 bit patterns (uint16 array) -> float64, exact."""
    h = np.ascontiguousarray(h).view(np.uint16)
    out = np.empty(h.shape, dtype=np.float64)
    _load().oracle_bf16_array_to_double(h.ctypes.data, out.ctypes.data, h.size)
    return out


def round_bf16_rne(x) -> np.ndarray:
    """float64 -> bfloat16 bit patterns (uint16), round to nearest, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_double_array_to_bf16_rne(x.ctypes.data, out.ctypes.data, x.size)
    return out
