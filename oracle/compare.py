"""Acceptance check of a GPU result against the oracle (test infrastructure).

Tolerances, elementwise, with ref and mag from the oracle
(mag = |alpha| * sum_k |a_ik b_kj| + |beta * C_in|):
  fp32:  |C - ref| <= 1e-5 * mag
  fp16:  |C - ref| <= 1e-4 * mag + 1e-3 * |ref| + 2^-25
         (the last two terms cover the final rounding of the fp32 result to
         fp16: at most 2^-11 |ref| for a normal result and half the spacing
         of the subnormals, 2^-24 / 2, below 2^-14)
  bf16:  |C - ref| <= 1e-4 * mag + 4e-3 * |ref| + 2^-134
         (bf16 keeps 8 significant bits: rounding the fp32 result moves it by
         at most 2^-9 |ref|, and the bound allows twice that; its subnormal
         spacing is 2^-133)
  small-integer inputs: bit-exact -- fp32 C == ref, fp16/bf16 C == RNE(ref).
The fp32 bound is the one the pages' observations support: reassociating an
fp32 sum moves low bits by ~1e-5 at 512^3 ("From a C loop to a GPU kernel",
"The benchmark is a trap too"); exactness holds whenever every partial sum is
representable ("The first loop" and the strict-k-order discussion).
"""
import numpy as np

from . import bf16_to_double, half_to_double, round_bf16_rne, round_half_rne

F32_REL = 1e-5
F16_REL = 1e-4
F16_OUT = 1e-3
BF16_OUT = 4e-3
F16_SUB = 2.0 ** -25   # half the spacing of binary16 subnormals
BF16_SUB = 2.0 ** -134  # half the spacing of bfloat16 subnormals


def as_double(C, dtype: str = None) -> np.ndarray:
    """Result array as float64; bfloat16 results come as uint16 bit patterns
    with dtype='bf16'."""
    C = np.asarray(C)
    if dtype == "bf16":
        return bf16_to_double(C)
    if C.dtype == np.float32:
        return C.astype(np.float64)
    if C.dtype in (np.float16, np.uint16):
        return half_to_double(C)
    if C.dtype == np.float64:
        return C
    raise TypeError(f"unexpected result dtype {C.dtype}")


def check(C, ref, mag, dtype: str, exact: bool = False) -> dict:
    """Compare result C (float32 or float16 array) with (ref, mag).

    Returns {"ok", "n", "bad", "worst_ratio", "max_abs_err"}; worst_ratio is
    max |C-ref| / bound (0/0 counts as 0, x/0 as inf).
    """
    ref = np.asarray(ref, dtype=np.float64)
    mag = np.asarray(mag, dtype=np.float64)
    Cd = as_double(C, dtype).reshape(ref.shape)
    err = np.abs(Cd - ref)
    if exact:
        if dtype in ("f16", "bf16"):
            want = round_half_rne(ref) if dtype == "f16" else round_bf16_rne(ref)
            got = np.ascontiguousarray(np.asarray(C)).view(np.uint16).reshape(ref.shape)
            bad = got != want
        else:
            bad = ~(Cd == ref)
        ratio = np.where(bad, np.inf, 0.0)
    else:
        if dtype == "f16":
            bound = F16_REL * mag + F16_OUT * np.abs(ref) + F16_SUB
        elif dtype == "bf16":
            bound = F16_REL * mag + BF16_OUT * np.abs(ref) + BF16_SUB
        else:
            bound = F32_REL * mag
        ok = err <= bound
        bad = ~ok
        with np.errstate(divide="ignore", invalid="ignore"):
            ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0),
                             np.where(err == 0, 0.0, np.inf))
        ratio = np.where(np.isnan(err), np.inf, ratio)
    nbad = int(np.count_nonzero(bad))
    return {
        "ok": nbad == 0,
        "n": int(ref.size),
        "bad": nbad,
        "worst_ratio": float(ratio.max()) if ratio.size else 0.0,
        "max_abs_err": float(np.nanmax(err)) if err.size and not np.all(np.isnan(err)) else
        (float("nan") if err.size else 0.0),
    }
