"""gemm_splitk_noalloc: the allocation-free entry point.

Some callers cannot allocate device memory at call time -- their allocator
already owns the GPU, or their process forbids allocation while serving.  For
them the library keeps the split-K partial sums in a fixed 8 MiB array.  This
test calls that entry point through the C ABI and checks that it gives the
same results as gemm() (within the tolerances the other tests use), on two
calls in a row so that whatever the first call left in the shared array cannot
leak into the second, and that a problem too large for the array is refused
before anything is launched.

The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from oracle import compare
from dense_gemm_tiled_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib(lib_path, gpu):
    from dense_gemm_tiled_gb300 import binding
    L = binding._lib
    i64, ci, cf, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
    L.gemm_splitk_noalloc.argtypes = [ci, ci, i64, i64, i64, ci, cf, cf, vp, i64, vp, i64, vp,
                                      i64, vp]
    L.gemm_splitk_noalloc.restype = ci
    return L, binding


def _call(L, p, A, B, C, stream):
    dt = 0 if p.dtype == "f32" else 1
    return L.gemm_splitk_noalloc(int(p.transA), int(p.transB), p.M, p.N, p.K, dt, p.alpha,
                                 p.beta, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
                                 C.data_ptr(), C.stride(0), stream)


@pytest.mark.parametrize("dtype,variant,shape", [
    ("f16", "nt", (512, 32, 5632)),   # LoRA adapter shapes: split-K path
    ("f16", "nn", (512, 32, 2048)),
    ("f32", "tn", (512, 32, 5632)),
    ("f16", "nt", (300, 520, 256)),   # no split: nothing in the array is used
])
def test_noalloc_matches_gemm_on_two_calls(lib, dtype, variant, shape):
    L, binding = lib
    M, N, K = shape
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream().cuda_stream
    for call, seed in enumerate((900, 901)):
        p = inputs.sweep_problem(M, N, K, variant, dtype, 0.5, seed=seed + 10 * M)
        A, B = p.A.to(dev), p.B.to(dev)
        C_ref = p.C_in.to(dev).clone()
        C_new = p.C_in.to(dev).clone()
        binding.gemm(A, B, C_ref, p.transA, p.transB, p.alpha, p.beta)
        rc = _call(L, p, A, B, C_new, stream)
        assert rc == 0, binding.status_string(rc)
        torch.cuda.synchronize()
        assert binding.check_device_status() == binding.OK
        # tolerance of the other tests, with gemm()'s output as the reference
        _, mag = oracle.gemm_ref(p.A.numpy(), p.B.numpy(), p.C_in.numpy(), p.transA, p.transB,
                                 p.alpha, p.beta)
        got = C_new.cpu().numpy()
        want = compare.as_double(C_ref.cpu().numpy())
        res = compare.check(got, want, mag, dtype)
        assert res["ok"], (call, res)


def test_noalloc_refuses_problems_larger_than_its_array(lib):
    L, binding = lib
    dev = torch.device("cuda:0")
    # a 512 x 512 fp16 output is 16 tiles of 128 x 128; with K = 8192 it is
    # split 9 ways: 9 MiB of fp32 partial sums, more than the 8 MiB array
    p = inputs.make_problem(512, 512, 8192, False, False, "f16", "uniform", seed=950)
    A, B = p.A.to(dev), p.B.to(dev)
    C = torch.full((512, 512), 7.0, dtype=torch.float16, device=dev)
    rc = _call(L, p, A, B, C, torch.cuda.current_stream().cuda_stream)
    assert rc == binding.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(C == 7.0)  # nothing was launched
