"""Pins of the oracle against facts that do not come from the oracle itself.

CPU only.  Each pin is chosen so that a plausible mistake in the oracle (a
dropped term, a wrong sign, a wrong or transposed index, a wrong fp16 exponent
bias, ties rounded the wrong way, a magnitude without absolute values) fails at
least one of them; test_pins_catch_planted_mistakes checks exactly that by
building broken copies of the oracle source and running the pins on them.
"""
import json
import os
import subprocess

import numpy as np
import pytest

import oracle
from oracle import compare

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_products.json")
VAR = {"nn": (False, False), "tn": (True, False), "nt": (False, True), "tt": (True, True)}


def _f32(x):
    return np.ascontiguousarray(np.array(x, dtype=np.float32))


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------
# pin functions (also run against planted-mistake builds)
# ---------------------------------------------------------------------------
def pin_hand_products(lib=None):
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        tA, tB = VAR[c["variant"]]
        Cin = _f32(c["C_in"]) if "C_in" in c else None
        ref, mag = oracle.gemm_ref(_f32(c["A"]), _f32(c["B"]), Cin, tA, tB, c["alpha"],
                                   c["beta"], lib=lib)
        assert np.array_equal(ref, np.array(c["C"], dtype=np.float64)), c["name"]
        assert np.array_equal(mag, np.array(c["mag"], dtype=np.float64)), c["name"]


def pin_integer_exact(lib=None):
    """Small-integer inputs: the result is an integer matrix computed exactly
    by numpy's int64 matmul (a library routine, independent of the oracle)."""
    r = _rng(1)
    for (M, N, K) in [(7, 5, 3), (17, 33, 5), (16, 9, 31)]:
        for v, (tA, tB) in VAR.items():
            A = r.integers(-3, 4, size=(K, M) if tA else (M, K))
            B = r.integers(-3, 4, size=(N, K) if tB else (K, N))
            C = r.integers(-3, 4, size=(M, N))
            opA = A.T if tA else A
            opB = B.T if tB else B
            want = 2 * (opA @ opB) + C  # alpha=2, beta=1, all integers
            ref, mag = oracle.gemm_ref(_f32(A), _f32(B), _f32(C), tA, tB, 2.0, 1.0, lib=lib)
            assert np.array_equal(ref, want.astype(np.float64)), (v, M, N, K)
            want_mag = 2 * (np.abs(opA) @ np.abs(opB)) + np.abs(C)
            assert np.array_equal(mag, want_mag.astype(np.float64)), (v, M, N, K)


def pin_transpose_identity(lib=None):
    """(AB)^T = B^T A^T ties the variants together: tn/nt/tt on transposed
    copies equal nn, and nn(B^T, A^T) is the transpose of nn(A, B)."""
    r = _rng(2)
    M, N, K = 6, 11, 9
    A = _f32(r.uniform(-1, 1, (M, K)))
    B = _f32(r.uniform(-1, 1, (K, N)))
    nn, _ = oracle.gemm_ref(A, B, lib=lib)
    At, Bt = np.ascontiguousarray(A.T), np.ascontiguousarray(B.T)
    assert np.array_equal(oracle.gemm_ref(At, B, transA=True, lib=lib)[0], nn)
    assert np.array_equal(oracle.gemm_ref(A, Bt, transB=True, lib=lib)[0], nn)
    assert np.array_equal(oracle.gemm_ref(At, Bt, transA=True, transB=True, lib=lib)[0], nn)
    swapped, _ = oracle.gemm_ref(Bt, At, lib=lib)
    assert np.array_equal(swapped, nn.T)


def pin_fp16_exhaustive(lib=None):
    """All 65536 binary16 patterns widen to the value numpy.float16 gives, and
    rounding that value back returns the same pattern."""
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = h.view(np.float16).astype(np.float64)
    l = lib or oracle._load()
    got = np.empty(65536, dtype=np.float64)
    l.oracle_half_array_to_double(h.ctypes.data, got.ctypes.data, h.size)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # signed zeros too
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))
    back = np.empty(65536, dtype=np.uint16)
    l.oracle_double_array_to_half_rne(got.ctypes.data, back.ctypes.data, got.size)
    assert np.array_equal(back[~nan], h[~nan])
    assert np.all(np.isnan(back[nan].view(np.float16)))


def pin_fp16_ties_to_even(lib=None):
    """Midpoints between adjacent finite binary16 values round to the one with
    an even significand, and arbitrary doubles round as numpy's RN-even cast."""
    l = lib or oracle._load()
    pos = np.arange(0, 0x7c00, dtype=np.uint32).astype(np.uint16)  # +0 .. max finite
    lo = pos[:-1].view(np.float16).astype(np.float64)
    hi = pos[1:].view(np.float16).astype(np.float64)
    mid = np.concatenate([(lo + hi) / 2, -(lo + hi) / 2])  # exact in double
    want = np.concatenate([np.where(pos[:-1] % 2 == 0, pos[:-1], pos[1:]),
                           np.where(pos[:-1] % 2 == 0, pos[:-1], pos[1:]) | 0x8000]).astype(np.uint16)
    got = np.empty(mid.size, dtype=np.uint16)
    l.oracle_double_array_to_half_rne(mid.ctypes.data, got.ctypes.data, mid.size)
    # -0.0 midpoint of (0, smallest subnormal) is -1.49e-8 -> rounds to -0 (0x8000)
    assert np.array_equal(got, want)
    x = _rng(3).normal(0, 1, 200000) * np.exp2(_rng(4).integers(-30, 18, 200000))
    got = np.empty(x.size, dtype=np.uint16)
    l.oracle_double_array_to_half_rne(x.ctypes.data, got.ctypes.data, x.size)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def pin_bf16_exhaustive(lib=None):
    """All 65536 bfloat16 patterns widen to the binary32 whose upper half they
    are (numpy's view of the bits), and rounding that value back returns the
    same pattern."""
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        want = (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    l = lib or oracle._load()
    got = np.empty(65536, dtype=np.float64)
    l.oracle_bf16_array_to_double(h.ctypes.data, got.ctypes.data, h.size)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))
    back = np.empty(65536, dtype=np.uint16)
    l.oracle_double_array_to_bf16_rne(got.ctypes.data, back.ctypes.data, got.size)
    assert np.array_equal(back[~nan], h[~nan])


def pin_bf16_ties_to_even(lib=None):
    """Midpoints between adjacent finite bfloat16 values round to the even
    pattern, and fp32 values round as torch's RN-even float32 -> bfloat16 cast."""
    import torch
    l = lib or oracle._load()
    pos = np.arange(0, 0x7f80, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        vals = (pos << 16).view(np.float32).astype(np.float64)
    mid = np.concatenate([(vals[:-1] + vals[1:]) / 2, -(vals[:-1] + vals[1:]) / 2])
    ev = np.where(pos[:-1] % 2 == 0, pos[:-1], pos[1:]).astype(np.uint16)
    want = np.concatenate([ev, ev | 0x8000]).astype(np.uint16)
    got = np.empty(mid.size, dtype=np.uint16)
    l.oracle_double_array_to_bf16_rne(mid.ctypes.data, got.ctypes.data, mid.size)
    assert np.array_equal(got, want)
    x = torch.randn(200000, generator=torch.Generator().manual_seed(5)) * \
        torch.exp2(torch.randint(-140, 120, (200000,), generator=torch.Generator().manual_seed(6)).float())
    x = x[torch.isfinite(x)]
    want = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xd = x.numpy().astype(np.float64)
    got = np.empty(xd.size, dtype=np.uint16)
    l.oracle_double_array_to_bf16_rne(xd.ctypes.data, got.ctypes.data, xd.size)
    assert np.array_equal(got, want)


def pin_bf16_integer_exact(lib=None):
    """bfloat16 small-integer operands: the oracle's product equals numpy's
    exact int64 matmul."""
    r = _rng(12)
    for v, (tA, tB) in VAR.items():
        A = r.integers(-3, 4, size=(9, 7) if tA else (7, 9))
        B = r.integers(-3, 4, size=(5, 9) if tB else (9, 5))
        as_bf16 = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        ref, _ = oracle.gemm_ref(as_bf16(A), as_bf16(B), None, tA, tB, lib=lib, fmt="bf16")
        want = (A.T if tA else A) @ (B.T if tB else B)
        assert np.array_equal(ref, want.astype(np.float64)), v


EPI_GOLDEN = os.path.join(os.path.dirname(GOLDEN), "epilogue_values.json")


def _bias_act(lib, x, bias, act):
    l = lib or oracle._load()
    x = np.array(x, dtype=np.float64)
    b = np.ascontiguousarray(bias, dtype=np.float64) if bias is not None else None
    assert l.oracle_bias_act(x.ctypes.data, x.shape[0], x.shape[1], x.shape[1],
                             None if b is None else b.ctypes.data, oracle.ACTS[act]) == 0
    return x


def pin_gelu_table(lib=None):
    """gelu(v) = v * Phi(v) against tabulated standard normal values, and the
    identity gelu(v) - gelu(-v) = v (Phi(v) + Phi(-v) = 1)."""
    l = lib or oracle._load()
    for v, want in json.load(open(EPI_GOLDEN))["gelu"]:
        got = l.oracle_gelu(v)
        assert abs(got - want) <= 1e-15 * max(1.0, abs(want)), (v, got, want)
    for v in np.linspace(-6, 6, 97):
        assert abs((l.oracle_gelu(v) - l.oracle_gelu(-v)) - v) <= 1e-14 * max(1.0, abs(v))
    # through the epilogue entry, with and without a bias
    x = np.array([[1.0, -1.0, 2.0]])
    got = _bias_act(lib, x, None, "gelu")
    assert np.allclose(got, [[0.8413447460685429, -0.15865525393145707, 1.9544997361036416]],
                       rtol=1e-15, atol=0)
    got = _bias_act(lib, x - 1.0, np.ones(3), "gelu")
    assert np.allclose(got, [[0.8413447460685429, -0.15865525393145707, 1.9544997361036416]],
                       rtol=1e-15, atol=0)


def pin_bias_per_column(lib=None):
    """The bias is a per-output (per-column) offset, added before the
    activation; relu is max(v, 0)."""
    g = json.load(open(EPI_GOLDEN))["bias_act"]
    for act in ("none", "relu"):
        got = _bias_act(lib, g["x"], g["bias"], act)
        assert np.array_equal(got, np.array(g[act])), (act, got)


PINS = [pin_hand_products, pin_integer_exact, pin_transpose_identity, pin_fp16_exhaustive,
        pin_fp16_ties_to_even, pin_bf16_exhaustive, pin_bf16_ties_to_even, pin_bf16_integer_exact,
        pin_gelu_table, pin_bias_per_column]


# ---------------------------------------------------------------------------
# the pins on the real oracle
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


def test_identity_and_permutation():
    r = _rng(5)
    A = _f32(r.uniform(-1, 1, (13, 13)))
    I = np.eye(13, dtype=np.float32)
    assert np.array_equal(oracle.gemm_ref(A, I)[0], A.astype(np.float64))
    assert np.array_equal(oracle.gemm_ref(I, A)[0], A.astype(np.float64))
    perm = r.permutation(13)
    P = np.ascontiguousarray(I[perm])  # P @ A picks rows perm of A
    assert np.array_equal(oracle.gemm_ref(P, A)[0], A[perm].astype(np.float64))
    assert np.array_equal(oracle.gemm_ref(A, np.ascontiguousarray(P.T))[0],
                          A[:, perm].astype(np.float64))


def test_numpy_float64_second_opinion():
    r = _rng(6)
    for v, (tA, tB) in VAR.items():
        M, N, K = 9, 14, 23
        A = _f32(r.uniform(-1, 1, (K, M) if tA else (M, K)))
        B = _f32(r.uniform(-1, 1, (N, K) if tB else (K, N)))
        C = _f32(r.uniform(-1, 1, (M, N)))
        opA = (A.T if tA else A).astype(np.float64)
        opB = (B.T if tB else B).astype(np.float64)
        want = 1.5 * opA @ opB - 0.75 * C.astype(np.float64)
        ref, mag = oracle.gemm_ref(A, B, C, tA, tB, 1.5, -0.75)
        assert np.allclose(ref, want, rtol=1e-12, atol=1e-12 * mag.max())


def test_fp16_operands_widen_exactly():
    r = _rng(7)
    A = r.uniform(-1, 1, (8, 12)).astype(np.float16)
    B = r.uniform(-1, 1, (12, 5)).astype(np.float16)
    ref, _ = oracle.gemm_ref(A, B)
    want = A.astype(np.float64) @ B.astype(np.float64)
    assert np.allclose(ref, want, rtol=1e-13, atol=1e-15)
    # integer fp16: exact
    Ai = r.integers(-3, 4, (8, 12)).astype(np.float16)
    Bi = r.integers(-3, 4, (12, 5)).astype(np.float16)
    assert np.array_equal(oracle.gemm_ref(Ai, Bi)[0],
                          (Ai.astype(np.int64) @ Bi.astype(np.int64)).astype(np.float64))


def test_alpha_beta_closed_forms():
    r = _rng(8)
    A = _f32(r.uniform(-1, 1, (5, 7)))
    B = _f32(r.uniform(-1, 1, (7, 6)))
    C = _f32(r.uniform(-1, 1, (5, 6)))
    ref, _ = oracle.gemm_ref(A, B, C, alpha=0.0, beta=-2.0)
    assert np.array_equal(ref, -2.0 * C.astype(np.float64))
    Cnan = np.full((5, 6), np.nan, dtype=np.float32)
    ref, mag = oracle.gemm_ref(A, B, Cnan, beta=0.0)
    assert np.all(np.isfinite(ref)) and np.all(np.isfinite(mag))


def test_zero_padding_invariance():
    """Embedding A and B in larger zero matrices leaves the product unchanged."""
    r = _rng(9)
    A = _f32(r.uniform(-1, 1, (10, 7)))
    B = _f32(r.uniform(-1, 1, (7, 12)))
    Ab = np.zeros((16, 19), np.float32); Ab[:10, :7] = A
    Bb = np.zeros((19, 21), np.float32); Bb[:7, :12] = B
    small, _ = oracle.gemm_ref(A, B)
    big, _ = oracle.gemm_ref(Ab, Bb)
    assert np.array_equal(big[:10, :12], small)
    assert np.all(big[10:, :] == 0) and np.all(big[:, 12:] == 0)


def test_leading_dimension_views():
    r = _rng(10)
    Abig = _f32(r.uniform(-1, 1, (9, 20)))
    Bbig = _f32(r.uniform(-1, 1, (11, 30)))
    A = Abig[:, :11]   # ld 20
    B = Bbig[:, :7]    # ld 30
    ref, _ = oracle.gemm_ref(A, B)
    ref2, _ = oracle.gemm_ref(np.ascontiguousarray(A), np.ascontiguousarray(B))
    assert np.array_equal(ref, ref2)


def test_points_equal_full():
    r = _rng(11)
    for v, (tA, tB) in VAR.items():
        M, N, K = 21, 17, 40
        A = _f32(r.uniform(-1, 1, (K, M) if tA else (M, K)))
        B = _f32(r.uniform(-1, 1, (N, K) if tB else (K, N)))
        C = _f32(r.uniform(-1, 1, (M, N)))
        ref, mag = oracle.gemm_ref(A, B, C, tA, tB, 0.5, 0.25)
        rows = r.integers(0, M, 50)
        cols = r.integers(0, N, 50)
        pr, pm = oracle.gemm_ref_points(A, B, rows, cols, C, tA, tB, 0.5, 0.25)
        assert np.array_equal(pr, ref[rows, cols])
        assert np.array_equal(pm, mag[rows, cols])


def test_k_zero_and_empty():
    C = _f32([[1, 2], [3, 4]])
    A = np.zeros((2, 0), np.float32)
    B = np.zeros((0, 2), np.float32)
    ref, mag = oracle.gemm_ref(A, B, C, beta=3.0)
    assert np.array_equal(ref, 3.0 * C.astype(np.float64))
    ref, _ = oracle.gemm_ref(np.zeros((0, 3), np.float32), np.zeros((3, 4), np.float32))
    assert ref.shape == (0, 4)


def test_checker_tolerances():
    ref = np.array([1.0, -2.0, 0.0])
    mag = np.array([10.0, 10.0, 0.0])
    ok = compare.check(np.array([1.00005, -2.0, 0.0], np.float32), ref, mag, "f32")
    assert ok["ok"]
    bad = compare.check(np.array([1.0002, -2.0, 0.0], np.float32), ref, mag, "f32")
    assert not bad["ok"] and bad["bad"] == 1
    nan = compare.check(np.array([np.nan, -2.0, 0.0], np.float32), ref, mag, "f32")
    assert not nan["ok"]
    ex = compare.check(np.array([2049.0, 3.0], np.float16), np.array([2049.0, 3.0]),
                       np.array([1.0, 1.0]), "f16", exact=True)
    # 2049 is not representable in fp16: RNE gives 2048, and float16(2049) is 2048 too
    assert ex["ok"]


def test_checker_subnormal_outputs():
    """A result below 2^-14 lands on fp16's subnormal grid (spacing 2^-24), so
    the correctly rounded value may sit up to 2^-25 from ref however small
    |ref| is; one whole quantum off must still fail.  Same for bfloat16 at its
    own subnormal spacing 2^-133."""
    q16 = 2.0 ** -24
    ref = np.array([1.0e-5 + 0.49 * q16, -3.0e-6 - 0.49 * q16])  # tiny single-term results
    mag = np.abs(ref)
    got = ref.astype(np.float16)  # numpy's RN-even cast onto the subnormal grid
    assert np.all(np.abs(got.astype(np.float64)) < 2.0 ** -14)
    assert compare.check(got, ref, mag, "f16")["ok"]
    off = (got.astype(np.float64) + np.array([q16, -q16])).astype(np.float16)
    assert compare.check(off, ref, mag, "f16")["bad"] == 2
    # bfloat16: values near 2^-130 (subnormal), given as uint16 bit patterns
    qb = 2.0 ** -133
    refb = np.array([37.1 * qb, -5.3 * qb])
    want = oracle.round_bf16_rne(refb)
    assert compare.check(want, refb, np.abs(refb), "bf16")["ok"]
    assert compare.check(want + np.uint16(1), refb, np.abs(refb), "bf16")["bad"] == 2


# ---------------------------------------------------------------------------
# planted mistakes: every one must trip at least one pin
# ---------------------------------------------------------------------------
MUTATIONS = {
    "dropped_last_k_term": ("for (int64_t k = 0; k < K; ++k) {          /* strict increasing k */",
                            "for (int64_t k = 0; k < K - 1; ++k) {"),
    "transA_ignored": ("return transA ? load_elem(A, dtype, k * lda + i)",
                       "return transA ? load_elem(A, dtype, i * lda + k)"),
    "transB_swapped_index": ("load_elem(B, dtype, k * ldb + j);",
                             "load_elem(B, dtype, j * ldb + k);"),
    "beta_wrong_sign": ("                r += j->beta * cin;\n                m += fabs(j->beta * cin);",
                        "                r -= j->beta * cin;\n                m += fabs(j->beta * cin);"),
    "mag_without_abs": ("macc[c] += fabs(p);", "macc[c] += p;"),
    "alpha_dropped": ("double r = j->alpha * acc[c];", "double r = acc[c];"),
    "fp16_bias_off_by_one": ("v = ldexp((double)(1024 + f), e - 25);",
                             "v = ldexp((double)(1024 + f), e - 24);"),
    "fp16_subnormal_scale": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "ties_away_from_zero": ("return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "return fl + 1.0;"),
    "rounding_truncates": ("if (d > 0.5) return fl + 1.0;", "if (d > 2.0) return fl + 1.0;"),
    "bf16_widen_shift": ("const uint32_t bits = (uint32_t)b << 16;",
                         "const uint32_t bits = (uint32_t)b << 15;"),
    "bf16_subnormal_scale": ("double r = rne_integer(ldexp(a, 133));",
                             "double r = rne_integer(ldexp(a, 132));"),
    "bf16_bias": ("return (uint16_t)(s | (uint16_t)((e + 127) << 7) | (uint16_t)((int)r - 128));",
                  "return (uint16_t)(s | (uint16_t)((e + 126) << 7) | (uint16_t)((int)r - 128));"),
    "bias_ignored": ("double v = x[i * ldx + j] + (bias ? bias[j] : 0.0);",
                     "double v = x[i * ldx + j];"),
    "bias_by_row": ("double v = x[i * ldx + j] + (bias ? bias[j] : 0.0);",
                    "double v = x[i * ldx + j] + (bias ? bias[i < cols ? i : 0] : 0.0);"),
    "relu_keeps_negatives": ("if (act == ORACLE_ACT_RELU) v = v > 0.0 ? v : 0.0;",
                             "if (act == ORACLE_ACT_RELU) v = v > 0.0 ? v : -v;"),
    "gelu_tanh_fit": ("double oracle_gelu(double v) { return 0.5 * v * (1.0 + erf(v / sqrt(2.0))); }",
                      "double oracle_gelu(double v) { return 0.5 * v * (1.0 + tanh(0.7978845608028654 * (v + 0.044715 * v * v * v))); }"),
    "gelu_missing_sqrt2": ("double oracle_gelu(double v) { return 0.5 * v * (1.0 + erf(v / sqrt(2.0))); }",
                           "double oracle_gelu(double v) { return 0.5 * v * (1.0 + erf(v / 2.0)); }"),
    "bf16_read_as_fp16": ("if (dtype == ORACLE_BF16) return oracle_bf16_to_double(((const uint16_t*)p)[idx]);",
                          "if (dtype == ORACLE_BF16) return oracle_half_to_double(((const uint16_t*)p)[idx]);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistakes(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle_gemm.c")).read()
    old, new = MUTATIONS[name]
    assert old in src, f"mutation target for {name} no longer in the oracle source"
    bad_src = tmp_path / "oracle_bad.c"
    bad_src.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_bad.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-pthread",
                    str(bad_src), "-o", str(so), "-lm"], check=True)
    lib = oracle.bind(str(so))
    failed = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name} passed every pin"


def test_checker_epilogue():
    """check_epilogue: the oracle's own bias/activation result, rounded to the
    output type, passes; a relative 1e-3 slip or a bias on the wrong axis
    fails."""
    r = _rng(9)
    ref = r.normal(0, 2, (6, 5))
    mag = np.abs(ref) * 4 + 1.0
    b = r.normal(0, 1, 5)
    for act in ("none", "relu", "gelu"):
        out = oracle.bias_act(ref, b, act)
        for dt, cast in (("f32", np.float32), ("f16", np.float16)):
            assert compare.check_epilogue(out.astype(cast), ref, mag, dt, b, act)["ok"], (act, dt)
        assert not compare.check_epilogue((out * 1.001 + 1e-3).astype(np.float32), ref, mag,
                                          "f32", b, act)["ok"]
    sq, msq = ref[:5], mag[:5]
    wrong_axis = oracle.bias_act(np.ascontiguousarray(sq.T), b, "none").T  # bias along rows
    assert not compare.check_epilogue(wrong_axis.astype(np.float32), sq, msq, "f32", b,
                                      "none")["ok"]


def _tf32(x, mode):
    """fp32 values reduced to TF32 (10 fraction bits) by truncation or by
    round-to-nearest-even of the low 13 bits, on the bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    if mode == "rne":
        lsb = (b >> 13) & 1
        b = b + 0xFFF + lsb
    b = (b & 0xFFFFE000) & 0xFFFFFFFF
    return b.astype(np.uint32).view(np.float32)


def test_tf32_bound_covers_operand_reduction():
    """The opt-in TF32 tolerance, (2^-9 + 1e-5) * mag, holds for a product of
    TF32-reduced operands -- truncated or rounded -- accumulated exactly, and
    is violated by a coarser (8 fraction bits) reduction; fp32's own bound is
    violated by TF32, so the tf32 check is the looser one it must be."""
    r = _rng(12)
    A = _f32(r.uniform(-1, 1, (64, 300)))
    B = _f32(r.uniform(-1, 1, (300, 48)))
    ref, mag = oracle.gemm_ref(A, B)
    for mode in ("trunc", "rne"):
        got = _tf32(A, mode).astype(np.float64) @ _tf32(B, mode).astype(np.float64)
        assert compare.check(got.astype(np.float32), ref, mag, "tf32")["ok"], mode
        assert not compare.check(got.astype(np.float32), ref, mag, "f32")["ok"], mode
    # same-signed operands make truncation errors add up: 10 kept fraction
    # bits stay inside the bound, 8 do not
    Ap, Bp = np.abs(A), np.abs(B)
    refp, magp = oracle.gemm_ref(Ap, Bp)
    got = _tf32(Ap, "trunc").astype(np.float64) @ _tf32(Bp, "trunc").astype(np.float64)
    assert compare.check(got.astype(np.float32), refp, magp, "tf32")["ok"]
    coarse = lambda x: (np.ascontiguousarray(x).view(np.uint32) & 0xFFFF8000).view(np.float32)
    got = coarse(Ap).astype(np.float64) @ coarse(Bp).astype(np.float64)
    assert not compare.check(got.astype(np.float32), refp, magp, "tf32")["ok"]
