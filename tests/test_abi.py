"""The C-ABI library: it builds, loads, exports every declared symbol, and
rejects bad arguments before touching the GPU (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(gemm[a-z_0-9]*)\s*\(",
                                 src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["gemm", "gemm_host", "gemm_check_device_status", "gemm_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


@pytest.fixture(scope="module")
def b(lib_path):
    from dense_gemm_tiled_gb300 import binding
    return binding


# fake, well-aligned, non-overlapping "device" addresses: argument checks never
# dereference them and no launch happens when a check fails
PA, PB, PC = 0x10000000, 0x20000000, 0x30000000


def test_status_strings(b):
    assert b.status_string(0) == "GEMM_OK"
    assert b.status_string(3) == "GEMM_ERR_ALIAS"
    assert b.status_string(99) == "GEMM_ERR_UNKNOWN"
    assert b.version() >> 16 == 1


@pytest.mark.parametrize("args,code", [
    # (transA, transB, M, N, K, dtype, A, lda, B, ldb, C, ldc)
    ((2, 0, 4, 4, 4, 0, PA, 4, PB, 4, PC, 4), 1),       # bad trans flag
    ((0, 0, 4, 4, 4, 7, PA, 4, PB, 4, PC, 4), 1),       # bad dtype
    ((0, 0, -1, 4, 4, 0, PA, 4, PB, 4, PC, 4), 1),      # negative M
    ((0, 0, 4, 4, 4, 0, PA, 3, PB, 4, PC, 4), 1),       # lda < K (nn)
    ((1, 0, 8, 4, 4, 0, PA, 4, PB, 4, PC, 4), 1),       # lda < M (tn)
    ((0, 1, 4, 8, 6, 0, PA, 6, PB, 5, PC, 8), 1),       # ldb < K (nt)
    ((0, 0, 4, 8, 4, 0, PA, 4, PB, 8, PC, 7), 1),       # ldc < N
    ((0, 0, 4, 4, 4, 0, 0, 4, PB, 4, PC, 4), 1),        # null A
    ((0, 0, 4, 4, 4, 0, PA, 4, PB, 4, 0, 4), 1),        # null C
    ((0, 0, 4, 4, 4, 0, PA + 2, 4, PB, 4, PC, 4), 1),   # misaligned fp32 A
    ((0, 0, 4, 4, 4, 1, PA + 1, 4, PB, 4, PC, 4), 1),   # misaligned fp16 A
    ((0, 0, 4, 4, 4, 0, PA, 4, PB, 4, PA + 16, 4), 3),  # C overlaps A
    ((0, 0, 4, 4, 4, 0, PA, 4, PB, 4, PB - 8, 4), 3),   # C overlaps B from below
    ((0, 0, 1 << 31, 4, 4, 0, PA, 4, PB, 4, PC, 4), 2),  # too large
])
def test_invalid_arguments(b, args, code):
    tA, tB, M, N, K, dt, A, lda, B, ldb, C, ldc = args
    assert b.gemm_raw(tA, tB, M, N, K, dt, 1.0, 0.0, A, lda, B, ldb, C, ldc) == code
    assert b.last_path() == "none"


def test_empty_output_returns_ok_without_gpu(b):
    assert b.gemm_raw(0, 0, 0, 5, 3, 0, 1.0, 0.0, PA, 3, PB, 5, PC, 5) == 0
    assert b.gemm_raw(0, 0, 5, 0, 3, 1, 1.0, 0.0, PA, 3, PB, 1, PC, 1) == 0
    assert b.gemm_raw(0, 0, 0, 0, 0, 0, 1.0, 0.0, 0, 1, 0, 1, 0, 1) == 0
    assert b.last_path() == "none"


@pytest.mark.parametrize("args,code", [
    # (M, N, K, dtype, A, lda, sA, B, ldb, sB, C, ldc, sC, batch), nn
    ((4, 4, 4, 0, PA, 4, 16, PB, 4, 16, PC, 4, 16, -1), 1),        # negative batch
    ((4, 4, 4, 0, PA, 4, -16, PB, 4, 16, PC, 4, 16, 2), 1),        # negative A pitch
    ((4, 4, 4, 0, PA, 4, 16, PB, 4, 16, PC, 4, -1, 2), 1),         # negative C pitch
    ((4, 4, 4, 0, PA, 4, 16, PB, 4, 16, PC, 4, 15, 2), 3),         # C entries overlap
    ((4, 4, 4, 0, PA, 4, 16, PB, 4, 16, PC, 4, 0, 3), 3),          # C pitch 0 (shared C)
    ((4, 4, 4, 0, PA, 4, 16, PB, 4, 16, PA + 64, 4, 16, 2), 3),    # C span meets A's 2nd entry
    ((4, 4, 4, 0, PA, 4, 0, PB, 4, 1 << 20, PB + 64, 4, 16, 2), 3),  # C inside B's span
    ((4, 4, 4, 0, PA, 3, 16, PB, 4, 16, PC, 4, 16, 2), 1),         # lda < K
    ((4, 4, 4, 0, PA, 4, 16, PB, 4, 16, PC, 4, 16, 1 << 31), 2),   # batch too large
    ((4, 4, 4, 0, PA, 4, 1 << 60, PB, 4, 16, PC, 4, 16, 64), 2),   # extent overflows
])
def test_batched_invalid_arguments(b, args, code):
    M, N, K, dt, A, lda, sA, B, ldb, sB, C, ldc, sC, batch = args
    assert b.gemm_strided_batched_raw(0, 0, M, N, K, dt, 1.0, 0.0, A, lda, sA, B, ldb, sB, C, ldc,
                                      sC, batch) == code
    assert b.last_path() == "none"


def test_batched_empty_returns_ok_without_gpu(b):
    assert b.gemm_strided_batched_raw(0, 0, 4, 4, 4, 0, 1.0, 0.0, PA, 4, 16, PB, 4, 16, PC, 4, 16,
                                      0) == 0
    assert b.gemm_strided_batched_raw(0, 0, 0, 4, 4, 1, 1.0, 0.0, PA, 4, 16, PB, 4, 16, PC, 4, 16,
                                      5) == 0
    assert b.last_path() == "none"


def test_gemm_ex_invalid_arguments(b):
    # (..., bias, act): bad act code, misaligned bias, bias overlapping C
    assert b.gemm_ex_raw(0, 0, 4, 4, 4, 0, 1.0, 0.0, PA, 4, PB, 4, PC, 4, 0, 3) == 1
    assert b.gemm_ex_raw(0, 0, 4, 4, 4, 0, 1.0, 0.0, PA, 4, PB, 4, PC, 4, PC + 4096 + 2, 1) == 1
    assert b.gemm_ex_raw(0, 0, 4, 4, 4, 0, 1.0, 0.0, PA, 4, PB, 4, PC, 4, PC + 16, 2) == 3
    assert b.gemm_ex_raw(0, 0, 0, 4, 4, 0, 1.0, 0.0, PA, 4, PB, 4, PC, 4, 0, 2) == 0
    assert b.last_path() == "none"


def test_tf32_not_accepted_without_scratch(b, lib_path):
    import ctypes
    lib = ctypes.CDLL(lib_path)
    f = lib.gemm_splitk_noalloc
    i64, ci, cf, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
    f.argtypes = [ci, ci, i64, i64, i64, ci, cf, cf, vp, i64, vp, i64, vp, i64, vp]
    f.restype = ci
    assert f(0, 0, 4, 4, 4, 3, 1.0, 0.0, PA, 4, PB, 4, PC, 4, None) == 2  # TF32
    assert f(0, 0, 4, 4, 4, 4, 1.0, 0.0, PA, 4, PB, 4, PC, 4, None) == 2  # 3xTF32
    assert b.gemm_raw(0, 0, 4, 4, 4, 5, 1.0, 0.0, PA, 4, PB, 4, PC, 4) == 1  # dtype 5 unknown


@pytest.mark.parametrize("entry", ["gemm", "gemm_strided_batched"])
def test_binding_refuses_host_tensors(lib_path, entry):
    """No CPU fallback: the device entry points refuse host tensors outright
    (host memory goes through gemm_host, whose copies are part of the call)."""
    import torch
    from dense_gemm_tiled_gb300 import binding
    shape = (4, 8, 8) if entry == "gemm_strided_batched" else (8, 8)
    A, B, C = torch.ones(shape), torch.ones(shape), torch.zeros(shape)
    with pytest.raises(ValueError):
        getattr(binding, entry)(A, B, C)
    assert torch.count_nonzero(C) == 0
