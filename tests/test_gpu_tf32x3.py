"""The opt-in 3xTF32 path (dtype GEMM_F32_3XTF32): fp32 operands split into
TF32 hi and lo parts, products hi*hi + hi*lo + lo*hi on kind::tf32 tensor-core
MMAs in one fp32 accumulation.  Checked against the oracle with the fp32
path's own tolerance (1e-5 * mag; the CPU model of the arithmetic in
test_tf32x3_model.py bounds the split's error by 2^-19 * mag), bit-exact on
small integers (lo = 0, every sum exact), and shown more accurate than plain
TF32 on the same inputs."""
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
    binding.gemm(A, B, C, prob.transA, prob.transB, prob.alpha, prob.beta, tf32x3=True, **kw)
    torch.cuda.synchronize()
    assert binding.check_device_status() == binding.OK
    return C.cpu(), binding.last_path()


def _check(prob, C, exact=False, seed=9):
    ref, mag, idx = oracle_for(prob, seed=seed)
    got = to_np(C)
    if idx is not None:
        got = got[idx[0], idx[1]]
    res = compare.check(got, ref, mag, "f32", exact=exact)
    assert res["ok"], f"{prob.name}: {res}"
    return res


@pytest.mark.parametrize("variant", ["nn", "tn", "nt", "tt"])
@pytest.mark.parametrize("shape", [(384, 640, 448), (300, 520, 264), (2048, 1536, 512),
                                   (1000, 3000, 777), (300, 523, 264),
                                   # few tiles, long K: shared (stream-K) tiles
                                   (256, 384, 6000)],
                         ids=lambda s: "x".join(map(str, s)))
def test_tf32x3_parity(variant, shape):
    M, N, K = shape
    beta = 0.5 if (M + K) % 2 == 0 else 0.0
    prob = inputs.sweep_problem(M, N, K, variant, "f32", beta, seed=850 + M)
    C, path = _run(prob)
    assert path in ("tc", "tc_splitk"), path
    _check(prob, C)


def test_tf32x3_normal_operands_4096():
    """The headline shape with weights-like and activation-like scales."""
    prob = inputs.make_problem(4096, 4096, 4096, False, False, "f32", "normal", seed=860,
                               std_a=1.0, std_b=0.02)
    C, _ = _run(prob)
    _check(prob, C, seed=3)


@pytest.mark.parametrize("variant", ["nn", "tn", "nt", "tt"])
def test_tf32x3_integer_exact(variant):
    tA, tB = inputs.VARIANTS[variant]
    prob = inputs.make_problem(320, 448, 384, tA, tB, "f32", "integer", seed=870, beta=1.0,
                               c_fill="integer")
    C, _ = _run(prob)
    _check(prob, C, exact=True)


def test_tf32x3_more_accurate_than_tf32():
    """On the same inputs plain TF32 leaves the fp32 bound and 3xTF32 meets it
    (so the lo terms really take part)."""
    from dense_gemm_tiled_gb300 import binding
    prob = inputs.sweep_problem(512, 512, 1024, "nn", "f32", 0.0, seed=880)
    ref, mag, _ = oracle_for(prob)
    A, B = prob.A.cuda(), prob.B.cuda()
    C1 = torch.empty((512, 512), dtype=torch.float32, device="cuda")
    binding.gemm(A, B, C1, tf32=True)
    C3 = torch.empty((512, 512), dtype=torch.float32, device="cuda")
    binding.gemm(A, B, C3, tf32x3=True)
    torch.cuda.synchronize()
    r1 = compare.check(to_np(C1.cpu()), ref, mag, "f32")
    r3 = compare.check(to_np(C3.cpu()), ref, mag, "f32")
    assert not r1["ok"] and r3["ok"]
    assert r3["worst_ratio"] < 0.25 * r1["worst_ratio"]


@pytest.mark.parametrize("act", ["relu", "gelu"])
def test_tf32x3_epilogue(act):
    prob = inputs.sweep_problem(1024, 768, 512, "nt", "f32", 0.0, seed=890)
    bias = inputs.uniform((768,), 891, "f32")
    C, _ = _run(prob, bias=bias.cuda(), act=act)
    ref, mag, _ = oracle_for(prob)
    res = compare.check_epilogue(to_np(C), ref, mag, "f32", to_np(bias).astype(np.float64), act)
    assert res["ok"], res
