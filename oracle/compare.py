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
  tf32:  |C - ref| <= (2^-9 + 1e-5) * mag   (the opt-in TF32 path keeps 10 of
         the 23 fraction bits of each operand: relative error below 2^-10 per
         operand, 2^-9 per product, plus the fp32 accumulation of fp32)
  small-integer inputs: bit-exact -- fp32 C == ref, fp16/bf16 C == RNE(ref).
The fp32 bound is the one the pages' observations support: reassociating an
fp32 sum moves low bits by ~1e-5 at 512^3 ("From a C loop to a GPU kernel",
"The benchmark is a trap too"); exactness holds whenever every partial sum is
representable ("The first loop" and the strict-k-order discussion).
"""
import numpy as np

from . import bf16_to_double, half_to_double, round_bf16_rne, round_half_rne

F32_REL = 1e-5
TF32_REL = 2.0 ** -9 + 1e-5
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
        elif dtype == "tf32":
            bound = TF32_REL * mag
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


GELU_LIPSCHITZ = 1.13  # max |d/dv v*Phi(v)| = 1.1289 (at v = sqrt(2))
EPI_ARITH = 2.0 ** -22  # the fp32 additions of alpha*acc, beta*C and the bias
GELU_EVAL = 2.0 ** -20  # fp32 evaluation of v/2 * (1 + erf(v / sqrt(2)))


def check_epilogue(C, ref_pre, mag, dtype: str, bias=None, act: str = "none", exact=False,
                   cols_index=None) -> dict:
    """Compare a fused-epilogue result C = act(alpha*AB + beta*C_in + bias[j])
    with the oracle ("From a C loop to a GPU kernel", section "Fusion").

    ref_pre, mag: the oracle's GEMM result and magnitude (before bias and
    activation); bias: float64 values per column or None; act: none, relu or
    gelu.  The bound propagates the GEMM bound through the activation (relu
    and identity are 1-Lipschitz, gelu 1.13-Lipschitz), adds the fp32
    rounding of the epilogue's additions and, for gelu, of its evaluation,
    then the output rounding of 16-bit results as check() does:
      bound = L * (rel(dtype) * mag + 2^-22 * (mag + |bias_j|))
              + [gelu] 2^-20 * (|x| + |out|) + out_rounding(dtype, |out|)
    with x = ref_pre + bias_j and out = act(x).  exact=True (small-integer
    inputs, identity or relu): C must equal out (fp32) or RNE(out)."""
    from . import bias_act
    ref_pre = np.asarray(ref_pre, dtype=np.float64)
    mag = np.asarray(mag, dtype=np.float64)
    out = bias_act(ref_pre, bias, act, cols_index=cols_index)
    if exact:
        return check(C, out, mag, dtype, exact=True)
    if bias is None:
        bj = np.zeros_like(ref_pre)
    else:
        b = np.asarray(bias, dtype=np.float64)
        bj = b[np.asarray(cols_index)] if ref_pre.ndim == 1 else np.broadcast_to(b, ref_pre.shape)
    x = ref_pre + bj
    rel = {"f32": F32_REL, "tf32": TF32_REL}.get(dtype, F16_REL)
    lip = GELU_LIPSCHITZ if act == "gelu" else 1.0
    bound = lip * (rel * mag + EPI_ARITH * (mag + np.abs(bj)))
    if act == "gelu":
        bound = bound + GELU_EVAL * (np.abs(x) + np.abs(out))
    if dtype == "f16":
        bound = bound + F16_OUT * np.abs(out) + F16_SUB
    elif dtype == "bf16":
        bound = bound + BF16_OUT * np.abs(out) + BF16_SUB
    Cd = as_double(C, dtype).reshape(out.shape)
    err = np.abs(Cd - out)
    bad = ~(err <= bound)
    nbad = int(np.count_nonzero(bad))
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / bound, np.where(err == 0, 0.0, np.inf))
    ratio = np.where(np.isnan(err), np.inf, ratio)
    return {"ok": nbad == 0, "n": int(out.size), "bad": nbad,
            "worst_ratio": float(ratio.max()) if ratio.size else 0.0,
            "max_abs_err": float(np.nanmax(err)) if err.size else 0.0}
