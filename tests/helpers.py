"""Shared test helpers: run a Problem through the C ABI and compare with the oracle."""
import numpy as np
import torch

import oracle
from oracle import compare

FULL_LIMIT = 1 << 33  # M*N*K up to this is checked element by element in full


def sample_points(M, N, seed, n_random=32768, corner=32):
    """Output positions for large problems: the first and last rows and columns,
    four corner blocks, the borders of the last (ragged) tile, and random points."""
    r = np.random.default_rng(seed)
    rows, cols = [], []
    for i in sorted({0, M - 1}):
        rows.append(np.full(N, i)); cols.append(np.arange(N))
    for j in sorted({0, N - 1}):
        rows.append(np.arange(M)); cols.append(np.full(M, j))
    for (r0, c0) in [(0, 0), (0, max(N - corner, 0)), (max(M - corner, 0), 0),
                     (max(M - corner, 0), max(N - corner, 0))]:
        rr, cc = np.meshgrid(np.arange(r0, min(r0 + corner, M)), np.arange(c0, min(c0 + corner, N)),
                             indexing="ij")
        rows.append(rr.ravel()); cols.append(cc.ravel())
    rows.append(r.integers(0, M, n_random)); cols.append(r.integers(0, N, n_random))
    return np.concatenate(rows).astype(np.int64), np.concatenate(cols).astype(np.int64)


def to_np(t: torch.Tensor) -> np.ndarray:
    """CPU numpy view; bfloat16 (no numpy dtype) comes back as uint16 bit
    patterns, which the oracle reads with fmt='bf16'."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def fmt_of(dtype: str):
    return "bf16" if dtype == "bf16" else None


def oracle_for(prob, full=None, seed=0):
    """(ref, mag, idx) with idx None for a full check or (rows, cols)."""
    A, B = to_np(prob.A), to_np(prob.B)
    C = to_np(prob.C_in) if prob.C_in is not None else None
    if full is None:
        full = prob.M * prob.N * max(prob.K, 1) <= FULL_LIMIT
    if full:
        ref, mag = oracle.gemm_ref(A, B, C, prob.transA, prob.transB, prob.alpha, prob.beta,
                                   fmt=fmt_of(prob.dtype))
        return ref, mag, None
    # fewer random points when each costs a K-long strided dot product
    n_random = 32768 if prob.K <= 4096 else 8192
    rows, cols = sample_points(prob.M, prob.N, seed, n_random=n_random)
    ref, mag = oracle.gemm_ref_points(A, B, rows, cols, C, prob.transA, prob.transB, prob.alpha,
                                      prob.beta, fmt=fmt_of(prob.dtype))
    return ref, mag, (rows, cols)


def run_gpu(prob, device="cuda:0", c_init=None):
    """Runs the product through the binding (C ABI) and returns C on the host."""
    from dense_gemm_tiled_gb300 import binding
    A = prob.A.to(device)
    B = prob.B.to(device)
    if prob.C_in is not None:
        C = prob.C_in.to(device).clone()
    elif c_init is not None:
        C = torch.full((prob.M, prob.N), c_init, dtype=prob.A.dtype, device=device)
    else:
        C = torch.empty((prob.M, prob.N), dtype=prob.A.dtype, device=device)
    binding.gemm(A, B, C, prob.transA, prob.transB, prob.alpha, prob.beta)
    torch.cuda.synchronize()
    assert binding.check_device_status() == binding.OK
    return C.cpu(), binding.last_path()


def check_problem(prob, exact=False, full=None, seed=0, c_init=None):
    C, path = run_gpu(prob, c_init=c_init)
    ref, mag, idx = oracle_for(prob, full, seed)
    got = to_np(C)
    if idx is not None:
        got = got[idx[0], idx[1]]
    res = compare.check(got, ref, mag, prob.dtype, exact=exact)
    res["path"] = path
    assert res["ok"], f"{prob.name}: {res}"
    return res
