"""bf16 operands / fp32 accumulate / bf16 output on the tcgen05 kernel, against
the oracle (bfloat16 widened exactly; tolerance 1e-4 * mag + 4e-3 * |ref|,
bit-exact RNE on small-integer inputs)."""
import pytest

from dense_gemm_tiled_gb300 import inputs
from helpers import check_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(lib_path, gpu):
    yield


@pytest.mark.parametrize("variant", ["nn", "tn", "nt", "tt"])
def test_one_tile_exact(variant):
    tA, tB = inputs.VARIANTS[variant]
    p = inputs.make_problem(128, 256, 64, tA, tB, "bf16", "integer", seed=1200)
    assert check_problem(p, exact=True)["path"] == "tc"


@pytest.mark.parametrize("variant", ["nn", "tn", "nt", "tt"])
def test_integer_exact_multi_tile(variant):
    tA, tB = inputs.VARIANTS[variant]
    p = inputs.make_problem(512, 768, 448, tA, tB, "bf16", "integer", seed=1201)
    check_problem(p, exact=True)


@pytest.mark.parametrize("variant", ["nn", "tn", "nt"])
def test_bf16_2048(variant):
    tA, tB = inputs.VARIANTS[variant]
    p = inputs.make_problem(2048, 2048, 2048, tA, tB, "bf16", "uniform", seed=1210)
    check_problem(p)


@pytest.mark.parametrize("N", [32, 64, 128, 200, 256, 328])
@pytest.mark.parametrize("variant", ["nn", "nt"])
def test_tile_widths(N, variant):
    p = inputs.sweep_problem(259, N, 200, variant, "bf16", 0.5, seed=1220 + N)
    check_problem(p)


@pytest.mark.parametrize("variant", ["nn", "tn", "nt"])
def test_unaligned_rows(variant):
    p = inputs.sweep_problem(1000, 3000, 777, variant, "bf16", 0.0, seed=1230)
    check_problem(p)


@pytest.mark.parametrize("shape", [(512, 32, 5632), (8192, 32, 8192)])
def test_skinny_split_k(shape):
    M, N, K = shape
    p = inputs.sweep_problem(M, N, K, "nt", "bf16", 0.5, seed=1240)
    assert check_problem(p)["path"] == "tc_splitk"


def test_lora_step_bf16():
    for i, g in enumerate(inputs.lora_step_gemms()):
        check_problem(inputs.lora_problem(g, seed=1300 + i, dtype="bf16"))
