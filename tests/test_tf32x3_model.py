"""The error bound of the opt-in 3xTF32 path, pinned on the CPU.

The path splits every fp32 operand value x into hi = x with the low 13
fraction bits cleared (its TF32 part) and lo = x - hi (exact in fp32), and
forms each product as hi(a) hi(b) + hi(a) lo(b) + lo(a) hi(b) on the tensor
cores, which read their operands as TF32.  This module models that arithmetic
in numpy -- the split, the TF32 reading of each operand (truncation, or
rounding to nearest: the model covers both), exact products and an exact sum
-- and checks it against the oracle: within 2^-19 * mag, which leaves the
fp32 tolerance (1e-5 * mag) room for the fp32 accumulation.  Planted
mistakes (one TF32 product only, either cross term dropped, lo not the
remainder of the hi actually used) must break the fp32 bound, so the pin is
not vacuous.
"""
import numpy as np
import pytest

import oracle
from oracle import compare
from dense_gemm_tiled_gb300 import inputs

MASK = np.uint32(0xFFFFE000)


def tf32_trunc(x):
    return (np.asarray(x, np.float32).view(np.uint32) & MASK).view(np.float32)


def tf32_round(x):
    """Round to nearest (ties away, the cvt.rna rule) at 10 fraction bits."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x1000)) & np.uint64(0xFFFFE000)
    return u.astype(np.uint32).view(np.float32)


def split(x):
    hi = tf32_trunc(x)
    lo = (np.asarray(x, np.float32) - hi).astype(np.float32)
    return hi, lo


def model(A, B, read, terms=("hh", "hl", "lh"), exact_lo=True):
    """Product of fp32 A [M,K], B [K,N] as the 3xTF32 path forms it, in double."""
    ah, al = split(A)
    bh, bl = split(B)
    if not exact_lo:  # a planted mistake: hi rounded, lo still the truncation's remainder
        ah, bh = tf32_round(A), tf32_round(B)
    f = lambda x: read(x).astype(np.float64)
    out = np.zeros((A.shape[0], B.shape[1]))
    if "hh" in terms:
        out += f(ah) @ f(bh)
    if "hl" in terms:
        out += f(ah) @ f(bl)
    if "lh" in terms:
        out += f(al) @ f(bh)
    return out


def _problems():
    yield inputs.make_problem(64, 48, 256, dtype="f32", dist="uniform", seed=41).A.numpy(), \
        inputs.make_problem(64, 48, 256, dtype="f32", dist="uniform", seed=41).B.numpy()
    p = inputs.make_problem(40, 72, 512, dtype="f32", dist="normal", seed=42, std_a=3.0,
                            std_b=0.02)
    yield p.A.numpy(), p.B.numpy()


@pytest.mark.parametrize("read", [tf32_trunc, tf32_round])
def test_model_within_fp32_bound(read):
    for A, B in _problems():
        ref, mag = oracle.gemm_ref(A, B)
        got = model(A, B, read)
        err = np.abs(got - ref)
        assert np.all(err <= 2.0 ** -19 * mag), float(np.max(err / mag))


@pytest.mark.parametrize("kind", ["hh", "no_hl", "no_lh", "mismatched_lo"])
def test_planted_mistakes_break_the_fp32_bound(kind):
    A, B = next(_problems())
    ref, mag = oracle.gemm_ref(A, B)
    if kind == "hh":
        got = model(A, B, tf32_trunc, terms=("hh",))
    elif kind == "no_hl":
        got = model(A, B, tf32_trunc, terms=("hh", "lh"))
    elif kind == "no_lh":
        got = model(A, B, tf32_trunc, terms=("hh", "hl"))
    else:
        got = model(A, B, tf32_trunc, exact_lo=False)
    assert not compare.check(got.astype(np.float32), ref, mag, "f32")["ok"]


def test_split_is_exact_and_small():
    x = inputs.uniform((4096,), 43, "f32").numpy() * np.float32(1e3)
    hi, lo = split(x)
    assert np.array_equal((hi.astype(np.float64) + lo.astype(np.float64)), x.astype(np.float64))
    assert np.all(np.abs(lo) <= 2.0 ** -10 * np.abs(x))
    assert np.all(tf32_trunc(hi) == hi)
