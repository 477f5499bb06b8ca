"""fp32 SGEMM (CUDA-core FFMA kernel) against the oracle."""
import pytest

from dense_gemm_tiled_gb300 import inputs
from helpers import check_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(lib_path, gpu):
    yield


def test_sgemm_512_uniform():
    res = check_problem(inputs.sgemm_512())
    assert res["path"] in ("ffma", "ffma_splitk")


def test_sgemm_512_integer_bit_exact():
    check_problem(inputs.sgemm_512(integer=True), exact=True)


@pytest.mark.parametrize("variant", ["nn", "tn", "nt", "tt"])
@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_variants_ragged(variant, beta):
    # several tiles in each direction plus ragged tails in M, N and K
    p = inputs.sweep_problem(300, 270, 131, variant, "f32", beta, seed=100)
    check_problem(p)


@pytest.mark.parametrize("variant", ["nn", "tn", "nt", "tt"])
def test_variants_integer_exact(variant):
    tA, tB = inputs.VARIANTS[variant]
    p = inputs.make_problem(257, 130, 200, tA, tB, "f32", "integer", seed=101, alpha=2.0,
                            beta=0.5, c_fill="integer")
    check_problem(p, exact=True)


@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 7, 3), (17, 33, 5), (127, 129, 130),
                                   (129, 127, 17), (1000, 3000, 777)])
def test_odd_shapes(shape):
    M, N, K = shape
    for i, v in enumerate(["nn", "tn", "nt"]):
        check_problem(inputs.sweep_problem(M, N, K, v, "f32", 0.0, seed=110 + i))


def test_sgemm_4096_sampled():
    check_problem(inputs.sgemm_4096(), full=False)


@pytest.mark.parametrize("shape", [(8192, 32, 8192), (512, 32, 5632), (32, 2048, 512)])
def test_skinny_split_k(shape):
    M, N, K = shape
    p = inputs.sweep_problem(M, N, K, "nn", "f32", 0.0, seed=120)
    res = check_problem(p)
    assert res["path"] == "ffma_splitk"


def test_skinny_split_k_beta():
    p = inputs.sweep_problem(512, 32, 5632, "tn", "f32", 0.5, seed=121)
    check_problem(p)


@pytest.mark.parametrize("shape", [(2048, 2048, 2048), (1000, 3000, 777), (1536, 1664, 4100),
                                   (1024, 1152, 4096)])
def test_stream_k_deterministic(shape):
    """Shapes whose tile count is not a whole number of rounds of the SMs run
    as one persistent launch whose last rounds share K steps between blocks
    (with fewer tiles than SMs, as 72 tiles at 1024 x 1152, every tile's);
    the block that finishes a shared tile adds the pieces in K order, so two
    runs agree bit for bit whichever block arrives last."""
    import torch
    from dense_gemm_tiled_gb300 import binding
    M, N, K = shape
    p = inputs.sweep_problem(M, N, K, "nn", "f32", 0.5, seed=130)
    r1 = check_problem(p, full=M * N * K <= (1 << 33))
    assert r1["path"] == "ffma"
    A, B = p.A.cuda(), p.B.cuda()
    outs = []
    for _ in range(3):
        C = p.C_in.cuda().clone()
        binding.gemm(A, B, C, False, False, p.alpha, p.beta)
        torch.cuda.synchronize()
        outs.append(C.cpu())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
