"""The fused epilogue (gemm_ex): C = act(alpha*op(A)op(B) + beta*C + bias[j]),
bias per output column, act none / relu / gelu ("From a C loop to a GPU
kernel", section "Fusion"), through every path of the library, against the
oracle's GEMM followed by its own bias/activation."""
import numpy as np
import pytest
import torch

import oracle
from oracle import compare
from dense_gemm_tiled_gb300 import inputs

from helpers import fmt_of, oracle_for, to_np

pytestmark = pytest.mark.gpu


def _bias(N, dtype, seed, integer=False):
    return (inputs.integers((N,), seed, dtype) if integer else inputs.uniform((N,), seed, dtype))


def _run(prob, bias, act):
    from dense_gemm_tiled_gb300 import binding
    A, B = prob.A.cuda(), prob.B.cuda()
    C = (prob.C_in.cuda().clone() if prob.C_in is not None
         else torch.full((prob.M, prob.N), float("nan"), dtype=prob.A.dtype, device="cuda"))
    binding.gemm(A, B, C, prob.transA, prob.transB, prob.alpha, prob.beta,
                 bias=None if bias is None else bias.cuda(), act=act)
    torch.cuda.synchronize()
    assert binding.check_device_status() == binding.OK
    return C.cpu(), binding.last_path()


def _check(prob, bias, act, exact=False, want_path=None):
    C, path = _run(prob, bias, act)
    if want_path:
        assert path == want_path, path
    ref, mag, idx = oracle_for(prob, seed=7)
    got = to_np(C)
    bd = None if bias is None else (oracle.bf16_to_double(to_np(bias)) if prob.dtype == "bf16"
                                    else to_np(bias).astype(np.float64))
    if idx is not None:
        got = got[idx[0], idx[1]]
        res = compare.check_epilogue(got, ref, mag, prob.dtype, bd, act, exact, cols_index=idx[1])
    else:
        res = compare.check_epilogue(got, ref, mag, prob.dtype, bd, act, exact)
    assert res["ok"], f"{prob.name} act={act}: {res}"


SHAPES = {
    # fp32: split-K (15 tiles), plain tiles, persistent stream-K with packing,
    # and rows of every operand off 16-byte alignment (odd leading dimensions:
    # operands copied to an aligned pitch first, C stored element-wise)
    "f32": [((300, 520, 1024), "ffma_splitk"), ((640, 1280, 64), "ffma"),
            ((1000, 2600, 620), "ffma"), ((1001, 2601, 621), "ffma")],
    # 16-bit: shared tiles (stream-K: 10 tiles, K = 6144), whole-K 2-SM pairs
    # (C stored by TMA, and loaded by TMA when beta != 0), and an odd N (C rows
    # off 16-byte alignment: stored through the staging buffers a row at a
    # time, or on a larger problem computed into an aligned copy that is then
    # copied into place)
    "f16": [((300, 520, 6144), "tc_splitk"), ((2048, 1536, 512), "tc"), ((2000, 1003, 512), None),
            ((2100, 1003, 512), None)],
    "bf16": [((300, 520, 6144), "tc_splitk"), ((2048, 1536, 512), "tc"),
             ((2000, 1003, 512), None)],
}


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("act", ["none", "relu", "gelu"])
@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_epilogue_paths(dtype, act, beta):
    for i, (shape, path) in enumerate(SHAPES[dtype]):
        M, N, K = shape
        for variant in ("nn", "nt"):
            prob = inputs.sweep_problem(M, N, K, variant, dtype, beta, seed=700 + i)
            prob.alpha = 0.75
            bias = _bias(N, dtype, 710 + i)
            _check(prob, bias, act, want_path=path)


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("act", ["relu", "gelu"])
def test_activation_without_bias(dtype, act):
    prob = inputs.sweep_problem(384, 640, 448, "tn", dtype, 0.0, seed=720)
    _check(prob, None, act)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_relu_bias_integer_exact(dtype):
    """Small-integer operands and an integer bias: relu(AB + bias) is exact."""
    prob = inputs.make_problem(256, 384, 192, False, True, dtype, "integer", seed=730, beta=1.0,
                               c_fill="integer")
    bias = _bias(384, dtype, 731, integer=True)
    _check(prob, bias, "relu", exact=True)


@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_epilogue_k_zero(dtype):
    """K == 0: C = act(beta * C + bias)."""
    from dense_gemm_tiled_gb300 import binding
    M, N = 70, 90
    C0 = inputs.uniform((M, N), 740, dtype)
    bias = _bias(N, dtype, 741)
    C = C0.cuda().clone()
    A = torch.empty((M, 0), dtype=C.dtype, device="cuda")
    B = torch.empty((0, N), dtype=C.dtype, device="cuda")
    binding.gemm(A, B, C, False, False, 1.0, 0.5, bias=bias.cuda(), act="gelu")
    torch.cuda.synchronize()
    assert binding.last_path() == "scale"
    ref = 0.5 * to_np(C0).astype(np.float64)
    res = compare.check_epilogue(to_np(C.cpu()), ref, np.abs(ref), dtype,
                                 to_np(bias).astype(np.float64), "gelu")
    assert res["ok"], res


def test_gelu_matches_definition_at_large_magnitudes():
    """gelu(v) -> v for large positive v and -> 0 for large negative v; the
    kernel's erff-based evaluation must not produce NaN or sign errors
    there (a 1 x N product with a single nonzero entry sets v directly)."""
    from dense_gemm_tiled_gb300 import binding
    v = torch.tensor([[-30.0, -8.0, -3.0, -0.5, 0.0, 0.5, 3.0, 8.0, 30.0]], dtype=torch.float32)
    A = torch.ones((1, 1), dtype=torch.float32, device="cuda")
    C = torch.empty((1, 9), dtype=torch.float32, device="cuda")
    binding.gemm(A, v.cuda(), C, act="gelu")
    torch.cuda.synchronize()
    got = C.cpu().numpy().astype(np.float64)[0]
    want = oracle.gelu(v.numpy().astype(np.float64)[0])
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - want) <= 2.0 ** -20 * (np.abs(v.numpy()[0]) + np.abs(want)) + 1e-30)
