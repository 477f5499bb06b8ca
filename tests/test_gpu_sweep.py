"""The shape sweep: squares 256 ... 8192 and the non-tile-multiple shapes
4095^3, 1000 x 3000 x 777 (rows not 16-byte aligned for fp16) and
8192 x 32 x 8192 (skinny: split-K), in fp32 and fp16, nn / tn / nt, with
beta = 0 and with beta = 0.5 on C ~ U[-1, 1).  Every output is checked against
the oracle up to 2^33 multiply-adds, sampled outputs above that (first and
last rows and columns, corner blocks, random points)."""
import pytest

from dense_gemm_tiled_gb300 import inputs
from helpers import check_problem

pytestmark = pytest.mark.gpu

SHAPES = [(n, n, n) for n in inputs.SWEEP_SQUARES] + inputs.SWEEP_ODD


@pytest.fixture(autouse=True)
def _lib(lib_path, gpu):
    yield


@pytest.mark.parametrize("variant", ["nn", "tn", "nt"])
@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_sweep(shape, dtype, variant):
    M, N, K = shape
    seed = 800 + SHAPES.index(shape) * 10 + ["nn", "tn", "nt"].index(variant)
    p = inputs.sweep_problem(M, N, K, variant, dtype, 0.5, seed=seed)
    check_problem(p, seed=seed)
    p0 = inputs.Problem(M, N, K, p.transA, p.transB, dtype, 1.0, 0.0, p.A, p.B, None,
                        p.name + "_b0")
    check_problem(p0, seed=seed)
