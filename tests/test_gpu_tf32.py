"""The opt-in TF32 path (dtype GEMM_F32_TF32): fp32 operands and output, products
on kind::tf32 tensor-core MMAs, against the oracle with the TF32 tolerance
(2^-9 + 1e-5) * mag, and bit-exact on small integers (exact in TF32)."""
import numpy as np
import pytest
import torch

from oracle import compare
from dense_gemm_tiled_gb300 import inputs

from helpers import oracle_for, to_np

pytestmark = pytest.mark.gpu


def _run(prob, **kw):
    from dense_gemm_tiled_gb300 import binding
    A, B = prob.A.cuda(), prob.B.cuda()
    C = (prob.C_in.cuda().clone() if prob.C_in is not None
         else torch.full((prob.M, prob.N), float("nan"), dtype=torch.float32, device="cuda"))
    binding.gemm(A, B, C, prob.transA, prob.transB, prob.alpha, prob.beta, tf32=True, **kw)
    torch.cuda.synchronize()
    assert binding.check_device_status() == binding.OK
    return C.cpu(), binding.last_path()


@pytest.mark.parametrize("variant", ["nn", "tn", "nt", "tt"])
@pytest.mark.parametrize("shape", [(384, 640, 448), (300, 520, 264), (2048, 1536, 512),
                                   (1000, 3000, 777),
                                   # odd N (C rows off 16-byte alignment): stored row
                                   # by row (small) or through an aligned copy (large)
                                   (300, 523, 264), (2100, 1003, 512)],
                         ids=lambda s: "x".join(map(str, s)))
def test_tf32_parity(variant, shape):
    M, N, K = shape
    beta = 0.5 if (M + K) % 2 == 0 else 0.0
    prob = inputs.sweep_problem(M, N, K, variant, "f32", beta, seed=800 + M)
    C, path = _run(prob)
    assert path in ("tc", "tc_splitk"), path
    ref, mag, idx = oracle_for(prob, seed=9)
    got = to_np(C)
    if idx is not None:
        got = got[idx[0], idx[1]]
    res = compare.check(got, ref, mag, "tf32")
    assert res["ok"], f"{prob.name}: {res}"


@pytest.mark.parametrize("variant", ["nn", "tn", "nt", "tt"])
def test_tf32_integer_exact(variant):
    """Integers in {-3..3} have at most 2 significant bits: exact in TF32, and
    every sum here is exact in fp32."""
    tA, tB = inputs.VARIANTS[variant]
    prob = inputs.make_problem(320, 448, 384, tA, tB, "f32", "integer", seed=810, beta=1.0,
                               c_fill="integer")
    C, _ = _run(prob)
    ref, mag, _ = oracle_for(prob)
    res = compare.check(to_np(C), ref, mag, "f32", exact=True)
    assert res["ok"], res


def test_tf32_is_reduced_precision():
    """The opt-in path really is TF32: on uniform inputs its error exceeds the
    fp32 path's bound somewhere (so the FFMA SGEMM is not being run instead),
    while the default fp32 path meets it."""
    from dense_gemm_tiled_gb300 import binding
    prob = inputs.sweep_problem(512, 512, 1024, "nn", "f32", 0.0, seed=820)
    C, path = _run(prob)
    assert path.startswith("tc")
    ref, mag, _ = oracle_for(prob)
    assert not compare.check(to_np(C), ref, mag, "f32")["ok"]
    A, B = prob.A.cuda(), prob.B.cuda()
    C2 = torch.empty((512, 512), dtype=torch.float32, device="cuda")
    binding.gemm(A, B, C2)
    torch.cuda.synchronize()
    assert binding.last_path().startswith("ffma")
    assert compare.check(to_np(C2.cpu()), ref, mag, "f32")["ok"]


@pytest.mark.parametrize("act", ["relu", "gelu"])
def test_tf32_epilogue(act):
    prob = inputs.sweep_problem(2048, 1536, 512, "nt", "f32", 0.0, seed=830)
    bias = inputs.uniform((1536,), 831, "f32")
    C, _ = _run(prob, bias=bias.cuda(), act=act)
    ref, mag, idx = oracle_for(prob, seed=4)
    got = to_np(C)
    if idx is not None:
        got = got[idx[0], idx[1]]
        res = compare.check_epilogue(got, ref, mag, "tf32", to_np(bias).astype(np.float64), act,
                                     cols_index=idx[1])
    else:
        res = compare.check_epilogue(got, ref, mag, "tf32", to_np(bias).astype(np.float64), act)
    assert res["ok"], res
