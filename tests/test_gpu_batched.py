"""Strided-batched GEMM and the attention product set against the oracle,
entry by entry ("Metal GEMM Kernels for LoRA Training on Apple Silicon",
section 8: per-head GEMMs entered at a head offset of a [H, N, d_h] tensor)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import compare
from dense_gemm_tiled_gb300 import inputs

from helpers import fmt_of, to_np

pytestmark = pytest.mark.gpu


def _oracle_entry(A, B, C_in, tA, tB, alpha, beta, dtype):
    return oracle.gemm_ref(to_np(A), to_np(B), None if C_in is None else to_np(C_in), tA, tB,
                           alpha, beta, fmt=fmt_of(dtype))


def _check_entries(C, A, B, C_in, tA, tB, alpha, beta, dtype, name, exact=False):
    C = C.cpu()
    for b in range(C.shape[0]):
        ref, mag = _oracle_entry(A[b], B[b], None if C_in is None else C_in[b], tA, tB, alpha, beta,
                                 dtype)
        res = compare.check(to_np(C[b]), ref, mag, dtype, exact=exact)
        assert res["ok"], f"{name} entry {b}: {res}"


def _run(prob, layout=None, device="cuda:0"):
    """Runs a BatchedProblem; `layout` optionally re-lays each operand out
    with padded row and batch pitches: {'A': (ld_pad, batch_pad), ...}."""
    from dense_gemm_tiled_gb300 import binding

    def place(t, key):
        t = t.to(device)
        if not layout or key not in layout:
            return t.contiguous()
        ld_pad, bpad = layout[key]
        bt, r, c = t.shape
        rows_total = r + bpad
        buf = torch.full((bt, rows_total, c + ld_pad), float("nan"), dtype=t.dtype, device=device)
        view = buf[:, :r, :c]
        view.copy_(t)
        return view

    A = place(prob.A, "A")
    B = place(prob.B, "B")
    if prob.C_in is not None:
        C = place(prob.C_in, "C")
    else:
        C = place(torch.zeros((prob.batch, prob.M, prob.N), dtype=prob.A.dtype), "C")
        if layout and "C" in layout:
            C.fill_(float("nan"))  # beta == 0: C is write-only
    binding.gemm_strided_batched(A, B, C, prob.transA, prob.transB, prob.alpha, prob.beta)
    torch.cuda.synchronize()
    assert binding.check_device_status() == binding.OK
    return C, binding.last_path(), binding.last_launches()


BATCH_CASES = [
    # (M, N, K, batch): several tiles, ragged tails, a batch spanning more
    # units than the persistent grid has blocks
    (200, 136, 72, 3),
    (256, 512, 192, 5),
    (136, 72, 104, 7),
    (384, 256, 128, 40),
]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("variant", ["nn", "tn", "nt", "tt"])
@pytest.mark.parametrize("shape", BATCH_CASES, ids=lambda s: "x".join(map(str, s)))
def test_batched_parity(dtype, variant, shape):
    M, N, K, batch = shape
    beta = 0.5 if (M + batch) % 2 else 0.0
    prob = inputs.batched_problem(M, N, K, batch, variant, dtype, seed=M + N + K + batch, beta=beta,
                                  alpha=1.25)
    C, path, launches = _run(prob)
    assert path == ("ffma_batched" if dtype == "f32" else "tc_batched"), path
    assert launches == 1
    _check_entries(C, prob.A, prob.B, prob.C_in, prob.transA, prob.transB, prob.alpha, prob.beta,
                   dtype, prob.name)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_batched_integer_exact(dtype):
    prob = inputs.batched_problem(160, 96, 128, 6, "nt", dtype, dist="integer", seed=3, beta=1.0)
    C, path, _ = _run(prob)
    _check_entries(C, prob.A, prob.B, prob.C_in, prob.transA, prob.transB, 1.0, 1.0, dtype,
                   prob.name, exact=True)


@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_batched_padded_pitches(dtype):
    """Row pitch above the row length and batch pitch above one matrix, for
    every operand; NaN in the gaps must not reach the result."""
    prob = inputs.batched_problem(136, 200, 96, 4, "nn", dtype, seed=8, beta=0.0)
    lay = {"A": (8, 3), "B": (16, 1), "C": (8, 5)}
    C, path, launches = _run(prob, layout=lay)
    assert path == ("ffma_batched" if dtype == "f32" else "tc_batched")
    _check_entries(C, prob.A, prob.B, None, False, False, 1.0, 0.0, dtype, prob.name)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("shared", ["A", "B"])
def test_batched_shared_operand(dtype, shared):
    """A batch pitch of 0 shares one matrix across the batch (a weight applied
    to every entry)."""
    from dense_gemm_tiled_gb300 import binding
    M, N, K, batch = 192, 320, 160, 5
    prob = inputs.batched_problem(M, N, K, batch, "nt", dtype, seed=21)
    A = prob.A.cuda()
    B = prob.B.cuda()
    if shared == "A":
        A = A[:1].expand(batch, -1, -1)
    else:
        B = B[:1].expand(batch, -1, -1)
    C = torch.empty((batch, M, N), dtype=A.dtype, device="cuda")
    binding.gemm_strided_batched(A, B, C, False, True)
    torch.cuda.synchronize()
    assert binding.check_device_status() == binding.OK
    assert binding.last_launches() == 1
    _check_entries(C, A.cpu(), B.cpu(), None, False, True, 1.0, 0.0, dtype, f"shared {shared}")


def test_batched_unaligned_runs_per_entry():
    """fp16 rows that are not 16-byte aligned (K = 100 in an nn A) cannot be
    described to the tensor-memory-access unit; the batch then runs entry by
    entry through the padded single-GEMM path, with the same results."""
    prob = inputs.batched_problem(150, 130, 100, 3, "nn", "f16", seed=5, beta=0.5)
    C, path, launches = _run(prob)
    assert path == "per_entry"
    assert launches >= 3
    _check_entries(C, prob.A, prob.B, prob.C_in, False, False, 1.0, 0.5, "f16", prob.name)


@pytest.mark.parametrize("dtype", ["f16", "f32"])
def test_batched_k_zero_scales_every_entry(dtype):
    from dense_gemm_tiled_gb300 import binding
    batch, M, N = 4, 33, 47
    C0 = inputs.uniform((batch, M, N), 9, dtype).cuda()
    C = C0.clone()
    A = torch.empty((batch, M, 0), dtype=C.dtype, device="cuda")
    B = torch.empty((batch, 0, N), dtype=C.dtype, device="cuda")
    binding.gemm_strided_batched(A, B, C, False, False, 1.0, 0.5)
    torch.cuda.synchronize()
    want = (C0.double().cpu() * 0.5)
    assert torch.equal(C.cpu().double(), want.to(C.dtype).double())


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("H,n,d", [(4, 256, 64), (16, 512, 64), (2, 200, 80)])
def test_attention_products(dtype, H, n, d):
    """The six GEMMs of one attention head's forward and backward pass, all
    heads in one batched call each, against the oracle per head."""
    from dense_gemm_tiled_gb300 import binding
    t = inputs.attention_tensors(H, n, d, seed=H + n + d, dtype=dtype)
    dev = {k: v.cuda() for k, v in t.items()}
    size = {"n": n, "d": d}
    for name, variant, left, right, Ms, Ns, Ks in inputs.ATTENTION_PRODUCTS:
        tA, tB = inputs.VARIANTS[variant]
        M, N = size[Ms], size[Ns]
        C = torch.empty((H, M, N), dtype=dev[left].dtype, device="cuda")
        binding.gemm_strided_batched(dev[left], dev[right], C, tA, tB)
        torch.cuda.synchronize()
        assert binding.check_device_status() == binding.OK
        if dtype != "f32" and d % 8 == 0:
            assert binding.last_path() == "tc_batched", (name, binding.last_path())
        _check_entries(C, t[left], t[right], None, tA, tB, 1.0, 0.0, dtype, f"{name} H{H} n{n} d{d}")


def test_attention_head_offset_is_a_plain_gemm():
    """Entry h of a batched call equals gemm() on the head's own matrix (the
    head offset of the section-8 layout), bit for bit."""
    from dense_gemm_tiled_gb300 import binding
    H, n, d = 6, 384, 64
    t = inputs.attention_tensors(H, n, d, seed=2, dtype="f16")
    Q, K = t["Q"].cuda(), t["K"].cuda()
    S = torch.empty((H, n, n), dtype=Q.dtype, device="cuda")
    binding.gemm_strided_batched(Q, K, S, False, True)
    for h in range(H):
        Sh = torch.empty((n, n), dtype=Q.dtype, device="cuda")
        binding.gemm(Q[h], K[h], Sh, False, True)
        torch.cuda.synchronize()
        assert torch.equal(Sh.view(torch.int16), S[h].view(torch.int16)), h


@pytest.mark.parametrize("dtype", ["f16", "f32"])
def test_attention_interleaved_heads(dtype):
    """Heads interleaved in a token-major [n, H, d] tensor: head h starts d
    elements after head h-1 and rows are H*d apart (batch pitch below one
    matrix).  The result must not depend on how the library runs it."""
    from dense_gemm_tiled_gb300 import binding
    H, n, d = 4, 256, 64
    Qt = inputs.normal((n, H, d), 77, 1.0, dtype)
    Kt = inputs.normal((n, H, d), 78, 1.0, dtype)
    Q = Qt.cuda().permute(1, 0, 2)  # [H, n, d] view, strides (d, H*d, 1)
    K = Kt.cuda().permute(1, 0, 2)
    S = torch.empty((H, n, n), dtype=Q.dtype, device="cuda")
    binding.gemm_strided_batched(Q, K, S, False, True)
    torch.cuda.synchronize()
    assert binding.check_device_status() == binding.OK
    _check_entries(S, Qt.permute(1, 0, 2).contiguous(), Kt.permute(1, 0, 2).contiguous(), None,
                   False, True, 1.0, 0.0, dtype, "interleaved QK^T")
