"""fp16 -> fp32-accumulate -> fp16 GEMM (tcgen05 kernel) against the oracle."""
import pytest

from dense_gemm_tiled_gb300 import inputs
from helpers import check_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(lib_path, gpu):
    yield


@pytest.mark.parametrize("variant", ["nn", "tn", "nt", "tt"])
def test_one_tile(variant):
    # a single 128 x 256 tile with one K block: the smallest complete path
    tA, tB = inputs.VARIANTS[variant]
    p = inputs.make_problem(128, 256, 64, tA, tB, "f16", "integer", seed=200)
    res = check_problem(p, exact=True)
    assert res["path"] == "tc"


@pytest.mark.parametrize("variant", ["nn", "tn", "nt", "tt"])
def test_integer_bit_exact_multi_tile(variant):
    tA, tB = inputs.VARIANTS[variant]
    p = inputs.make_problem(384, 640, 448, tA, tB, "f16", "integer", seed=201)
    check_problem(p, exact=True)


@pytest.mark.parametrize("variant", ["nn", "tn", "nt"])
def test_hgemm_2048(variant):
    res = check_problem(inputs.hgemm_square(2048, variant))
    assert res["path"] == "tc"


@pytest.mark.parametrize("N", [32, 48, 64, 96, 128, 200, 256, 328])
@pytest.mark.parametrize("variant", ["nn", "tn", "nt"])
def test_tile_widths(N, variant):
    # every BN configuration, with ragged M, N and K
    p = inputs.sweep_problem(259, N, 200, variant, "f16", 0.0, seed=210 + N)
    check_problem(p)


@pytest.mark.parametrize("variant", ["nn", "tn", "nt"])
def test_beta(variant):
    p = inputs.sweep_problem(300, 520, 260, variant, "f16", 0.5, seed=220)
    check_problem(p)


@pytest.mark.parametrize("variant", ["nn", "tn", "nt"])
def test_unaligned_rows_repacked(variant):
    # K = 777: fp16 rows of 1554 bytes, not 16-byte aligned -> padded copies
    p = inputs.sweep_problem(1000, 3000, 777, variant, "f16", 0.0, seed=230)
    check_problem(p)


@pytest.mark.parametrize("shape", [(512, 32, 5632), (8192, 32, 8192), (512, 32, 4096)])
def test_skinny_split_k(shape):
    M, N, K = shape
    p = inputs.sweep_problem(M, N, K, "nn", "f16", 0.0, seed=240)
    res = check_problem(p)
    assert res["path"] == "tc_splitk"


def test_skinny_split_k_integer_exact():
    p = inputs.make_problem(512, 32, 5632, False, True, "f16", "integer", seed=241)
    res = check_problem(p, exact=True)
    assert res["path"] == "tc_splitk"


@pytest.mark.parametrize("shape", [(8192, 32, 8192), (1024, 1024, 8192), (2048, 3072, 1024)])
def test_stream_k_deterministic(shape):
    """Shared tiles are summed in K order whichever contributor arrives last,
    so repeated calls give identical bits."""
    import torch
    from dense_gemm_tiled_gb300 import binding
    M, N, K = shape
    p = inputs.make_problem(M, N, K, False, False, "f16", "uniform", seed=243)
    A, B = p.A.cuda(), p.B.cuda()
    outs = []
    for _ in range(3):
        C = torch.empty((M, N), dtype=torch.float16, device="cuda")
        binding.gemm(A, B, C)
        outs.append(C)
    torch.cuda.synchronize()
    assert binding.check_device_status() == binding.OK
    assert all(torch.equal(outs[0], o) for o in outs[1:])
