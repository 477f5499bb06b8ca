"""Thin Python binding over libgemm_gb300.so (include/gemm.h).

Argument marshalling only: every step of the GEMM runs in the library's
kernels.  PyTorch supplies device memory and the current CUDA stream.  If the
library has not been built this module raises ImportError; there is no
fallback implementation.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgemm_gb300.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`"
        " or `python -m dense_gemm_tiled_gb300.build`")

_lib = ctypes.CDLL(LIB_PATH)

_i64, _int, _flt, _vp = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
_GEMM_ARGS = [_int, _int, _i64, _i64, _i64, _int, _flt, _flt, _vp, _i64, _vp, _i64, _vp, _i64,
              _vp]
_lib.gemm.argtypes = _GEMM_ARGS
_lib.gemm.restype = _int
_lib.gemm_ex.argtypes = _GEMM_ARGS[:-1] + [_vp, _int, _vp]
_lib.gemm_ex.restype = _int
_lib.gemm_host.argtypes = _GEMM_ARGS
_lib.gemm_host.restype = _int
_lib.gemm_strided_batched.argtypes = [_int, _int, _i64, _i64, _i64, _int, _flt, _flt, _vp, _i64,
                                      _i64, _vp, _i64, _i64, _vp, _i64, _i64, _i64, _vp]
_lib.gemm_strided_batched.restype = _int
_lib.gemm_check_device_status.argtypes = [_vp]
_lib.gemm_check_device_status.restype = _int
_lib.gemm_status_string.argtypes = [_int]
_lib.gemm_status_string.restype = ctypes.c_char_p
_lib.gemm_version.restype = _int
_lib.gemm_last_path.restype = _int
_lib.gemm_last_launches.restype = _int
_lib.gemm_last_grid.restype = _int
_lib.gemm_total_launches.restype = _i64
_lib.gemm_set_wait_timeout_ns.argtypes = [_i64]
_lib.gemm_set_wait_timeout_ns.restype = None
_lib.gemm_set_fault_injection.argtypes = [_int]
_lib.gemm_set_fault_injection.restype = None
_lib.gemm_set_kernel_events.argtypes = [_vp, _vp]
_lib.gemm_set_kernel_events.restype = None
_lib.gemm_scratch_high_water.argtypes = [_int]
_lib.gemm_scratch_high_water.restype = _i64

F32 = 0
F16_F32ACC = 1
BF16_F32ACC = 2
F32_TF32 = 3
F32_3XTF32 = 4
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALIAS, ERR_CUDA, ERR_NO_MEMORY, ERR_TIMEOUT = range(7)
PATHS = {0: "none", 1: "scale", 2: "ffma", 3: "ffma_splitk", 4: "tc", 5: "tc_splitk",
         6: "ffma_batched", 7: "tc_batched", 8: "per_entry"}


class GemmError(RuntimeError):
    def __init__(self, code: int):
        self.code = code
        super().__init__(status_string(code))


def status_string(code: int) -> str:
    return _lib.gemm_status_string(int(code)).decode()


def version() -> int:
    return _lib.gemm_version()


def last_path() -> str:
    return PATHS.get(_lib.gemm_last_path(), "unknown")


def last_launches() -> int:
    return _lib.gemm_last_launches()


def last_grid() -> int:
    return _lib.gemm_last_grid()


def total_launches() -> int:
    return _lib.gemm_total_launches()


def set_wait_timeout_ns(ns: int) -> None:
    _lib.gemm_set_wait_timeout_ns(int(ns))


def set_fault_injection(mode: int) -> None:
    _lib.gemm_set_fault_injection(int(mode))


def scratch_high_water(reset: bool = False) -> int:
    """Most bytes in use at once from the library's scratch pool on the
    current device since the last reset (0: none taken); reset=True then
    clears the mark."""
    return _lib.gemm_scratch_high_water(1 if reset else 0)


def set_kernel_events(start=None, end=None) -> None:
    """Brackets the main GEMM kernel of later calls on this thread with two
    torch.cuda.Event objects (each recorded once beforehand, so that its CUDA
    event exists); no arguments turns it off."""
    if start is None or end is None:
        _lib.gemm_set_kernel_events(None, None)
        return
    s, e = int(start.cuda_event), int(end.cuda_event)
    if not s or not e:
        raise ValueError("record each event once before passing it")
    _lib.gemm_set_kernel_events(s, e)


def gemm_raw(transA, transB, M, N, K, dtype, alpha, beta, A, lda, B, ldb, C, ldc,
             stream=0) -> int:
    """The C entry point with plain integers (device addresses, stream handle)."""
    return _lib.gemm(int(transA), int(transB), int(M), int(N), int(K), int(dtype), float(alpha),
                     float(beta), A or None, int(lda), B or None, int(ldb), C or None, int(ldc),
                     stream or None)


def gemm_ex_raw(transA, transB, M, N, K, dtype, alpha, beta, A, lda, B, ldb, C, ldc, bias, act,
                stream=0) -> int:
    """gemm_ex with plain integers (device addresses, act code)."""
    return _lib.gemm_ex(int(transA), int(transB), int(M), int(N), int(K), int(dtype),
                        float(alpha), float(beta), A or None, int(lda), B or None, int(ldb),
                        C or None, int(ldc), bias or None, int(act), stream or None)


def gemm_host_raw(transA, transB, M, N, K, dtype, alpha, beta, A, lda, B, ldb, C, ldc,
                  stream=0) -> int:
    """gemm_host with plain integers (host addresses)."""
    return _lib.gemm_host(int(transA), int(transB), int(M), int(N), int(K), int(dtype),
                          float(alpha), float(beta), A or None, int(lda), B or None, int(ldb),
                          C or None, int(ldc), stream or None)


def gemm_strided_batched_raw(transA, transB, M, N, K, dtype, alpha, beta, A, lda, strideA, B,
                             ldb, strideB, C, ldc, strideC, batch, stream=0) -> int:
    """gemm_strided_batched with plain integers (device addresses, element
    pitches, stream handle)."""
    return _lib.gemm_strided_batched(int(transA), int(transB), int(M), int(N), int(K), int(dtype),
                                     float(alpha), float(beta), A or None, int(lda), int(strideA),
                                     B or None, int(ldb), int(strideB), C or None, int(ldc),
                                     int(strideC), int(batch), stream or None)


def _ld3(t) -> int:
    """Row pitch of a [batch, rows, cols] tensor (the _ld rule per matrix)."""
    if t.shape[2] > 1 and t.stride(2) != 1:
        raise ValueError("rows must be contiguous (stride(2) == 1)")
    if t.shape[1] <= 1:
        return max(int(t.stride(1)), int(t.shape[2]), 1)
    return int(t.stride(1))


def gemm_strided_batched(A, B, C, transA=False, transB=False, alpha=1.0, beta=0.0, stream=None):
    """C[b] = alpha * op(A[b]) @ op(B[b]) + beta * C[b] for every b, in place.

    A, B, C are 3-D CUDA tensors [batch, rows, cols] with contiguous rows; the
    batch pitch is each tensor's stride(0) (0, via expand(), shares one A or
    B across the batch).  Shapes per entry as gemm().  Returns C.
    """
    import torch
    if A.dim() != 3 or B.dim() != 3 or C.dim() != 3:
        raise ValueError("batched operands are 3-D [batch, rows, cols]")
    batch = int(C.shape[0])
    if A.shape[0] != batch or B.shape[0] != batch:
        raise ValueError("A, B and C must have the same batch size")
    if A.dtype != B.dtype or A.dtype != C.dtype:
        raise TypeError("A, B and C must share a dtype")
    dtype = _DTYPES.get(A.dtype)
    if dtype is None:
        raise TypeError(f"unsupported dtype {A.dtype}")
    M, K = (A.shape[2], A.shape[1]) if transA else (A.shape[1], A.shape[2])
    Kb, N = (B.shape[2], B.shape[1]) if transB else (B.shape[1], B.shape[2])
    if K != Kb:
        raise ValueError(f"inner dimensions differ: {K} vs {Kb}")
    if C.shape[1] != M or C.shape[2] != N:
        raise ValueError(f"C is {tuple(C.shape)}, expected {(batch, M, N)}")
    if not (A.is_cuda and B.is_cuda and C.is_cuda):
        raise ValueError("gemm_strided_batched() takes CUDA tensors")
    s = stream if stream is not None else torch.cuda.current_stream(C.device)
    pitch = (lambda t: int(t.stride(0)) if batch > 1 else 0)
    rc = _lib.gemm_strided_batched(
        int(transA), int(transB), int(M), int(N), int(K), dtype, float(alpha), float(beta),
        A.data_ptr() or None, _ld3(A), pitch(A), B.data_ptr() or None, _ld3(B), pitch(B),
        C.data_ptr() or None, _ld3(C), pitch(C), batch, s.cuda_stream or None)
    if rc != OK:
        raise GemmError(rc)
    return C


def _ld(t) -> int:
    if t.dim() != 2:
        raise ValueError("matrices are 2-D")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError("rows must be contiguous (stride(1) == 1)")
    if t.shape[0] <= 1:  # a single row: any ld >= its length is valid
        return max(int(t.stride(0)), int(t.shape[1]), 1)
    return int(t.stride(0))


_DTYPES = {}


def _dtype_codes():
    import torch
    _DTYPES.update({torch.float32: F32, torch.float16: F16_F32ACC, torch.bfloat16: BF16_F32ACC})


def _dims(A, B, C, transA, transB):
    if A.dtype != B.dtype or A.dtype != C.dtype:
        raise TypeError("A, B and C must share a dtype")
    dtype = _DTYPES.get(A.dtype)
    if dtype is None:
        raise TypeError(f"unsupported dtype {A.dtype}")
    M, K = (A.shape[1], A.shape[0]) if transA else (A.shape[0], A.shape[1])
    Kb, N = (B.shape[1], B.shape[0]) if transB else (B.shape[0], B.shape[1])
    if K != Kb:
        raise ValueError(f"inner dimensions differ: {K} vs {Kb}")
    if tuple(C.shape) != (M, N):
        raise ValueError(f"C is {tuple(C.shape)}, expected {(M, N)}")
    return dtype, int(M), int(N), int(K)


ACTS = {"none": 0, "relu": 1, "gelu": 2}


def _current_stream(device_index: int) -> int:
    """Raw handle of the current CUDA stream of a device."""
    import torch
    get_raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if get_raw is not None:
        return get_raw(device_index)
    return torch.cuda.current_stream(device_index).cuda_stream


def _ld_of(shape, stride) -> int:
    """_ld from a 2-D shape and stride already fetched."""
    if shape[1] > 1 and stride[1] != 1:
        raise ValueError("rows must be contiguous (stride(1) == 1)")
    if shape[0] <= 1:
        return max(stride[0], shape[1], 1)
    return stride[0]


def gemm(A, B, C, transA=False, transB=False, alpha=1.0, beta=0.0, stream=None, bias=None,
         act="none", tf32=False, tf32x3=False):
    """C = act(alpha * op(A) @ op(B) + beta * C + bias) in place, on torch CUDA
    tensors.

    A is [M,K] (or [K,M] with transA), B is [K,N] (or [N,K] with transB),
    C is [M,N]; all float32, all float16 or all bfloat16 (fp32 accumulation), rows
    contiguous, any leading dimension.  bias: None or a contiguous CUDA tensor
    of N elements of C's dtype (per output column); act: 'none', 'relu' or
    'gelu'.  tf32=True (float32 tensors only) opts into the reduced-precision
    TF32 tensor-core path; tf32x3=True into the 3xTF32 tensor-core path (about
    fp32 accuracy, finite inputs).  Runs on `stream` (a torch.cuda.Stream) or
    the current stream.  Returns C.
    """
    dt = A.dtype
    dtype = _DTYPES.get(dt)
    if dtype is None or B.dtype != dt or C.dtype != dt:
        if B.dtype != dt or C.dtype != dt:
            raise TypeError("A, B and C must share a dtype")
        raise TypeError(f"unsupported dtype {dt}")
    sa, sb, sc = A.shape, B.shape, C.shape
    if len(sa) != 2 or len(sb) != 2 or len(sc) != 2:
        raise ValueError("matrices are 2-D")
    M, K = (sa[1], sa[0]) if transA else (sa[0], sa[1])
    Kb, N = (sb[1], sb[0]) if transB else (sb[0], sb[1])
    if K != Kb:
        raise ValueError(f"inner dimensions differ: {K} vs {Kb}")
    if sc[0] != M or sc[1] != N:
        raise ValueError(f"C is {tuple(sc)}, expected {(M, N)}")
    if tf32 or tf32x3:
        if dtype != F32 or (tf32 and tf32x3):
            raise TypeError("tf32=True or tf32x3=True (one of them) takes float32 tensors")
        dtype = F32_TF32 if tf32 else F32_3XTF32
    if not (A.is_cuda and B.is_cuda and C.is_cuda):
        raise ValueError("gemm() takes CUDA tensors; use gemm_host() for host memory")
    s = stream.cuda_stream if stream is not None else _current_stream(C.get_device())
    lda, ldb, ldc = _ld_of(sa, A.stride()), _ld_of(sb, B.stride()), _ld_of(sc, C.stride())
    if bias is not None or act != "none":
        if bias is not None:
            if not bias.is_cuda or bias.dtype != C.dtype or bias.numel() != N or \
                    not bias.is_contiguous():
                raise ValueError("bias: a contiguous CUDA tensor of N elements of C's dtype")
        rc = _lib.gemm_ex(int(transA), int(transB), M, N, K, dtype, float(alpha), float(beta),
                          A.data_ptr() or None, lda, B.data_ptr() or None, ldb,
                          C.data_ptr() or None, ldc,
                          (bias.data_ptr() or None) if bias is not None else None, ACTS[act],
                          s or None)
        if rc != OK:
            raise GemmError(rc)
        return C
    rc = _gemm_fn(int(transA), int(transB), M, N, K, dtype, float(alpha), float(beta),
                  A.data_ptr() or None, lda, B.data_ptr() or None, ldb, C.data_ptr() or None,
                  ldc, s or None)
    if rc != OK:
        raise GemmError(rc)
    return C


_gemm_fn = _lib.gemm


def gemm_host(A, B, C, transA=False, transB=False, alpha=1.0, beta=0.0, stream=None):
    """The same product on host (CPU) tensors, pinned or not; the library
    copies them to the GPU, computes, copies C back and synchronises."""
    import torch
    dtype, M, N, K = _dims(A, B, C, transA, transB)
    for t in (A, B, C):
        if t.is_cuda:
            raise ValueError("gemm_host() takes host tensors")
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = _lib.gemm_host(int(transA), int(transB), M, N, K, dtype, float(alpha), float(beta),
                        A.data_ptr() or None, _ld(A), B.data_ptr() or None, _ld(B),
                        C.data_ptr() or None, _ld(C), s.cuda_stream or None)
    if rc != OK:
        raise GemmError(rc)
    return C


def check_device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status:
    OK, ERR_TIMEOUT (a kernel's bounded wait ran out) or ERR_CUDA."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return _lib.gemm_check_device_status(s.cuda_stream or None)


try:
    _dtype_codes()
except ImportError:  # pragma: no cover - torch is needed only by the tensor wrappers
    pass
