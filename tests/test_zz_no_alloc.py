"""gemm_splitk_noalloc: the allocation-free entry point.

Some callers cannot allocate device memory at call time -- their allocator
already owns the GPU, or their process forbids allocation while serving.  For
them the library keeps the partial sums it would otherwise take from its
scratch pool in a fixed 8 MiB array.  This test calls that entry point through
the C ABI and checks, on two calls in a row (so that whatever the first call
left in the shared array cannot leak into the second):
  - each result against the oracle, at the tolerances the other tests use, or
    bit for bit on small-integer inputs;
  - that the shapes meant to split K did take a split path;
  - that the second call allocated nothing: the device's free memory, torch's
    allocator and the library's scratch pool are unchanged across it (the
    first call, made before any gemm() on the shape, has loaded the kernels);
  - that a problem too large for the array is refused before anything runs.
gemm() on the same inputs is checked against the oracle as a second check.

The file name makes pytest collect it last.
"""
import ctypes

import pytest
import torch

from dense_gemm_tiled_gb300 import inputs
from helpers import oracle_for, to_np
from oracle import compare

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


def _problem(dtype, variant, shape, dist, seed):
    M, N, K = shape
    tA, tB = inputs.VARIANTS[variant]
    if dist == "integer":
        return inputs.make_problem(M, N, K, tA, tB, dtype, "integer", seed=seed)
    return inputs.make_problem(M, N, K, tA, tB, dtype, "uniform", seed=seed, beta=0.5)


SPLIT_PATHS = ("tc_splitk", "ffma_splitk")


@pytest.mark.parametrize("dtype,variant,shape,dist,split", [
    ("f16", "nt", (512, 32, 5632), "uniform", True),   # LoRA adapter shapes: shared K
    ("f16", "nn", (512, 32, 4096), "uniform", True),
    ("f16", "nt", (512, 32, 5632), "integer", True),   # bit-exact through the shared tiles
    ("f32", "tn", (512, 32, 5632), "uniform", True),   # narrow fp32 tile, split K
    ("f32", "nn", (1000, 32, 3000), "integer", True),
    ("f16", "nt", (300, 520, 256), "uniform", False),  # whole tiles: the array is not used
])
def test_noalloc_matches_oracle_on_two_calls(lib, dtype, variant, shape, dist, split):
    L, binding = lib
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream().cuda_stream
    probs = [_problem(dtype, variant, shape, dist, seed=900 + 10 * call + shape[0])
             for call in range(2)]
    # every tensor exists before the first call, so nothing below allocates
    # through torch
    dev_in = [(p.A.to(dev), p.B.to(dev), p.C_in.to(dev).clone() if p.C_in is not None else
               torch.zeros((p.M, p.N), dtype=p.A.dtype, device=dev)) for p in probs]
    C_gemm = [c.clone() for (_, _, c) in dev_in]
    torch.cuda.synchronize()
    for call, (p, (A, B, C)) in enumerate(zip(probs, dev_in)):
        if call == 1:
            free0 = torch.cuda.mem_get_info()[0]
            torch0 = torch.cuda.memory_allocated()
            assert binding.scratch_high_water(reset=True) >= 0
        rc = _call(L, p, A, B, C, stream)
        assert rc == 0, binding.status_string(rc)
        path = binding.last_path()
        torch.cuda.synchronize()
        assert binding.check_device_status() == binding.OK
        if call == 1:
            assert torch.cuda.mem_get_info()[0] == free0
            assert torch.cuda.memory_allocated() == torch0
            assert binding.scratch_high_water() == 0
        assert (path in SPLIT_PATHS) == split, path
        ref, mag, _ = oracle_for(p, full=True)
        res = compare.check(to_np(C.cpu()), ref, mag, dtype, exact=(dist == "integer"))
        assert res["ok"], (call, res)
    # second check: gemm() on the same inputs, after the no-alloc calls
    for p, (A, B, _), C in zip(probs, dev_in, C_gemm):
        binding.gemm(A, B, C, p.transA, p.transB, p.alpha, p.beta)
        torch.cuda.synchronize()
        ref, mag, _ = oracle_for(p, full=True)
        res = compare.check(to_np(C.cpu()), ref, mag, dtype, exact=(dist == "integer"))
        assert res["ok"], res


def test_noalloc_refuses_problems_larger_than_its_array(lib):
    L, binding = lib
    dev = torch.device("cuda:0")
    # a 1152 x 1152 fp32 output is 81 tiles of 128 x 128, split over K (4096)
    # on any GPU with at least 81 SMs; one slice of partial sums is already
    # 1152 * 1152 * 4 bytes = 5.3 MB, so two or more exceed the 8 MiB array
    p = inputs.make_problem(1152, 1152, 4096, False, False, "f32", "uniform", seed=950)
    A, B = p.A.to(dev), p.B.to(dev)
    C = torch.full((1152, 1152), 7.0, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    rc = _call(L, p, A, B, C, torch.cuda.current_stream().cuda_stream)
    assert rc == binding.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(C == 7.0)  # nothing was launched
