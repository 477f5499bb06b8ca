"""Edge behaviour through the C ABI: beta == 0 never reads C, guard bands around
C stay untouched, K == 0, sub-matrix views, host buffers, and the bounded wait
reporting a timeout instead of hanging."""
import numpy as np
import pytest
import torch

import oracle
from oracle import compare
from dense_gemm_tiled_gb300 import inputs
from helpers import check_problem, fmt_of, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(lib_path, gpu):
    yield


def _b():
    from dense_gemm_tiled_gb300 import binding
    return binding


@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_beta_zero_ignores_nan_in_c(dtype):
    p = inputs.sweep_problem(200, 300, 100, "nn", dtype, 0.0, seed=300)
    check_problem(p, c_init=float("nan"))


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("variant", ["nn", "tn", "nt"])
def test_guard_bands_untouched(dtype, variant):
    """C lives inside a larger buffer (ldc > N, rows above and below); every
    element outside the M x N window must keep its sentinel."""
    b = _b()
    M, N, K = 131, 257, 70
    p = inputs.sweep_problem(M, N, K, variant, dtype, 0.5, seed=310)
    dt = inputs.DTYPES[dtype]
    pad_r, pad_c = 8, 24
    sentinel = 1234.0  # exactly representable in fp32 and fp16
    big = torch.full((M + 2 * pad_r, N + pad_c), sentinel, dtype=dt, device="cuda")
    C = big[pad_r:pad_r + M, :N]
    C.copy_(p.C_in.cuda())
    b.gemm(p.A.cuda(), p.B.cuda(), C, p.transA, p.transB, p.alpha, p.beta)
    torch.cuda.synchronize()
    host = big.cpu().float().numpy()
    mask = np.ones(host.shape, dtype=bool)
    mask[pad_r:pad_r + M, :N] = False
    assert np.all(host[mask] == sentinel)
    ref, mag = oracle.gemm_ref(to_np(p.A), to_np(p.B), to_np(p.C_in), p.transA, p.transB,
                               p.alpha, p.beta)
    res = compare.check(to_np(C.cpu()), ref, mag, dtype)
    assert res["ok"], res


@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_k_zero_scales_c(dtype):
    b = _b()
    dt = inputs.DTYPES[dtype]
    A = torch.empty((64, 0), dtype=dt, device="cuda")
    B = torch.empty((0, 48), dtype=dt, device="cuda")
    C0 = inputs.uniform((64, 48), 320, dtype)
    C = C0.cuda().clone()
    b.gemm(A, B, C, beta=0.5)
    torch.cuda.synchronize()
    assert b.last_path() == "scale"
    assert torch.equal(C.cpu(), (C0.float() * 0.5).to(dt))
    b.gemm(A, B, C, beta=0.0)
    torch.cuda.synchronize()
    assert torch.count_nonzero(C).item() == 0


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("variant", ["nn", "tn", "nt"])
def test_submatrix_views(dtype, variant):
    """Operands entered at an offset inside larger buffers (lda, ldb, ldc larger
    than the rows), as the LoRA page's row-split enters A and C by offset."""
    b = _b()
    tA, tB = inputs.VARIANTS[variant]
    M, N, K = 150, 210, 96
    dt = inputs.DTYPES[dtype]
    Abig = inputs.uniform((400, 400), 330, dtype)
    Bbig = inputs.uniform((400, 400), 331, dtype)
    ar, ac = (K, M) if tA else (M, K)
    br, bc = (N, K) if tB else (K, N)
    A = Abig[16:16 + ar, 8:8 + ac]
    B = Bbig[24:24 + br, 32:32 + bc]
    Cbig = torch.zeros((M + 10, N + 40), dtype=dt, device="cuda")
    C = Cbig[5:5 + M, 8:8 + N]
    b.gemm(Abig.cuda()[16:16 + ar, 8:8 + ac], Bbig.cuda()[24:24 + br, 32:32 + bc], C, tA, tB)
    torch.cuda.synchronize()
    ref, mag = oracle.gemm_ref(A.numpy(), B.numpy(), None, tA, tB)
    res = compare.check(to_np(C.cpu()), ref, mag, dtype)
    assert res["ok"], res


@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_gemm_host_buffers(dtype):
    b = _b()
    p = inputs.sweep_problem(300, 200, 150, "nt", dtype, 0.5, seed=340)
    A = p.A.pin_memory()
    B = p.B.pin_memory()
    C = p.C_in.clone().pin_memory()
    b.gemm_host(A, B, C, p.transA, p.transB, p.alpha, p.beta)
    ref, mag = oracle.gemm_ref(to_np(p.A), to_np(p.B), to_np(p.C_in), p.transA, p.transB,
                               p.alpha, p.beta)
    res = compare.check(to_np(C), ref, mag, dtype)
    assert res["ok"], res
    # pageable memory too
    C2 = p.C_in.clone()
    b.gemm_host(p.A, p.B, C2, p.transA, p.transB, p.alpha, p.beta)
    assert torch.equal(C2, C)


def test_bounded_wait_reports_timeout_and_context_survives():
    """A load that never arrives (test hook): the kernel's wait runs out after
    its limit, the status word says so, and the next call works."""
    b = _b()
    p = inputs.make_problem(256, 256, 512, False, False, "f16", "integer", seed=350)
    A, B = p.A.cuda(), p.B.cuda()
    C = torch.zeros((256, 256), dtype=torch.float16, device="cuda")
    assert b.check_device_status() == b.OK
    b.set_wait_timeout_ns(100_000_000)  # 0.1 s
    b.set_fault_injection(1)
    try:
        b.gemm(A, B, C)
        assert b.check_device_status() == b.ERR_TIMEOUT
    finally:
        b.set_fault_injection(0)
        b.set_wait_timeout_ns(0)
    assert b.check_device_status() == b.OK  # cleared by the read
    b.gemm(A, B, C)
    assert b.check_device_status() == b.OK
    ref, mag = oracle.gemm_ref(to_np(p.A), to_np(p.B))
    assert compare.check(to_np(C.cpu()), ref, mag, "f16", exact=True)["ok"]


def test_bounded_wait_reports_timeout_fp32_tma_staging():
    """The same for the fp32 kernel whose operand tiles arrive by TMA (tn:
    both operands stored k-major; 192 output tiles, no K split)."""
    b = _b()
    p = inputs.make_problem(2048, 1536, 256, True, False, "f32", "integer", seed=351)
    A, B = p.A.cuda(), p.B.cuda()
    C = torch.zeros((2048, 1536), dtype=torch.float32, device="cuda")
    assert b.check_device_status() == b.OK
    b.set_wait_timeout_ns(100_000_000)  # 0.1 s
    b.set_fault_injection(1)
    try:
        b.gemm(A, B, C, True, False)
        assert b.last_path() == "ffma"
        assert b.check_device_status() == b.ERR_TIMEOUT
    finally:
        b.set_fault_injection(0)
        b.set_wait_timeout_ns(0)
    assert b.check_device_status() == b.OK
    b.gemm(A, B, C, True, False)
    assert b.check_device_status() == b.OK
    ref, mag = oracle.gemm_ref(to_np(p.A), to_np(p.B), None, True, False)
    assert compare.check(to_np(C.cpu()), ref, mag, "f32", exact=True)["ok"]


def test_kernel_events_bracket_the_gemm_kernel():
    """gemm_set_kernel_events: the library records the caller's events around
    its main kernel only, so on a problem with a packing pre-pass (fp32 nn
    above the packing threshold) the kernel's time is positive and below the
    whole call's."""
    import torch
    from dense_gemm_tiled_gb300 import binding
    p = inputs.sweep_problem(2048, 2048, 2048, "nn", "f32", 0.0, seed=140)
    A, B = p.A.cuda(), p.B.cuda()
    C = torch.empty((2048, 2048), dtype=torch.float32, device="cuda")
    ks, ke = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ks.record(); ke.record()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    binding.set_kernel_events(ks, ke)
    try:
        for _ in range(3):
            s0.record()
            binding.gemm(A, B, C)
            s1.record()
            s1.synchronize()
    finally:
        binding.set_kernel_events()
    call_ms, kernel_ms = s0.elapsed_time(s1), ks.elapsed_time(ke)
    assert 0.0 < kernel_ms < call_ms, (kernel_ms, call_ms)
    # turned off: the events are no longer re-recorded
    before = ks.elapsed_time(ke)
    binding.gemm(A, B, C)
    torch.cuda.synchronize()
    assert ks.elapsed_time(ke) == before


@pytest.mark.parametrize("dtype,variant,M", [("f32", "nn", 1024), ("f32", "tn", 1000),
                                             ("f32", "nt", 4096), ("f32", "nt", 2048),
                                             ("f16", "tn", 1000), ("bf16", "nn", 2048)])
def test_gemm_host_pipelined(dtype, variant, M):
    """gemm_host on problems of at least 2^30 multiply-adds runs row panels of
    C on the device while later panels' A rows are still arriving and earlier
    panels' C rows are leaving (two copy streams); with fp32 and K >= 1024 the
    first panel runs over K slices as B arrives.  Every panel must match the
    oracle, beta included."""
    b = _b()
    N, K = 1536, 1024 if M < 4096 else 256
    p = inputs.sweep_problem(M, N, K, variant, dtype, 0.5, seed=345)
    A, B = p.A.pin_memory(), p.B.pin_memory()
    C = p.C_in.clone().pin_memory()
    b.gemm_host(A, B, C, p.transA, p.transB, p.alpha, p.beta)
    full = M * N * K <= (1 << 31)
    from helpers import oracle_for
    ref, mag, idx = oracle_for(p, full=full, seed=3)
    got = to_np(C)
    if idx is not None:
        got = got[idx[0], idx[1]]
    res = compare.check(got, ref, mag, dtype)
    assert res["ok"], res


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("shape", [(256, 256, 2048), (1024, 768, 512)], ids=["splitk", "whole"])
@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
def test_dependent_calls_back_to_back(dtype, shape, graph):
    """Calls queued on one stream with no synchronisation between them, each
    reading what the one before wrote (Y2 = Y1 W2 after Y1 = X W1) or
    overwriting what it read (Y1 = X' W1 after Y2 read Y1): the library's
    kernels may start while the previous one runs, so each must wait for it
    before touching memory.  Split-K shapes add the reduction kernel to the
    chain.  Eager and captured in a CUDA graph, against the oracle."""
    b = _b()
    M, N, K = shape  # Y1 [M, K] feeds the second product, which is [M, K] x [K, N]
    X = inputs.uniform((M, K), 900, dtype)
    X2 = inputs.uniform((M, K), 901, dtype)
    W1 = inputs.uniform((K, K), 902, dtype)
    W2 = inputs.uniform((K, N), 903, dtype)
    d = {k: v.cuda() for k, v in dict(X=X, X2=X2, W1=W1, W2=W2).items()}
    Y1 = torch.empty((M, K), dtype=d["X"].dtype, device="cuda")
    Y2 = torch.empty((M, N), dtype=d["X"].dtype, device="cuda")
    s = torch.cuda.Stream()

    def chain():
        b.gemm(d["X"], d["W1"], Y1, stream=s)
        b.gemm(Y1, d["W2"], Y2, stream=s)
        b.gemm(d["X2"], d["W1"], Y1, stream=s)

    with torch.cuda.stream(s):
        chain()
    s.synchronize()
    if graph:
        Y1.fill_(float("nan"))
        Y2.fill_(float("nan"))
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            chain()
        g.replay()
        torch.cuda.synchronize()
    assert b.check_device_status() == b.OK
    fmt = fmt_of(dtype)
    ref1, mag1 = oracle.gemm_ref(to_np(X2), to_np(W1), None, False, False, 1.0, 0.0, fmt=fmt)
    assert compare.check(to_np(Y1.cpu()), ref1, mag1, dtype)["ok"]
    # the second product is checked on the operand it read: the first Y1,
    # recomputed alone (the library is deterministic) and itself checked
    Y1a = torch.empty_like(Y1)
    b.gemm(d["X"], d["W1"], Y1a)
    torch.cuda.synchronize()
    r0, m0 = oracle.gemm_ref(to_np(X), to_np(W1), None, False, False, 1.0, 0.0, fmt=fmt)
    assert compare.check(to_np(Y1a.cpu()), r0, m0, dtype)["ok"]
    ref2, mag2 = oracle.gemm_ref(to_np(Y1a.cpu()), to_np(W2), None, False, False, 1.0, 0.0,
                                 fmt=fmt)
    assert compare.check(to_np(Y2.cpu()), ref2, mag2, dtype)["ok"]
