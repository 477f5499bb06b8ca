"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random numbers; it holds none of the GEMM arithmetic.
Every draw happens on the CPU with a torch.Generator seeded explicitly, so the
same (shape, seed) gives the same bits within one PyTorch build.  Across builds
(another version or CPU architecture) the vectorised normal transform may
differ in the last bit, so a test draws its inputs in the process that runs
both the GPU path and the oracle, and no stored expected value depends on
these draws.

Distributions (the workloads' own descriptions; the pages name no generator,
so torch's CPU generator is the reading taken):
  uniform   i.i.d. U[-1, 1): torch.rand * 2 - 1 in fp32 (exact), then rounded
            (RN-even) to fp16 or bf16 for 16-bit operands.
  integer   i.i.d. integers in {-3..3}: exact in fp32, fp16 and bf16, so
            every product and every partial sum at these sizes is exact.
  normal    N(0, std^2) in fp32, then rounded to the operand type: weights
            std 0.02, activations std 1 (the LoRA MLP-block set).
"""
from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def uniform(shape, seed: int, dtype: str = "f32") -> torch.Tensor:
    x = torch.rand(tuple(shape), generator=_gen(seed), dtype=torch.float32) * 2.0 - 1.0
    return x.to(DTYPES[dtype])


def integers(shape, seed: int, dtype: str = "f32", lo: int = -3, hi: int = 3) -> torch.Tensor:
    x = torch.randint(lo, hi + 1, tuple(shape), generator=_gen(seed), dtype=torch.int32)
    return x.to(DTYPES[dtype])


def normal(shape, seed: int, std: float = 1.0, dtype: str = "f32") -> torch.Tensor:
    x = torch.randn(tuple(shape), generator=_gen(seed), dtype=torch.float32) * float(std)
    return x.to(DTYPES[dtype])


def draw(dist: str, shape, seed: int, dtype: str, std: float = 1.0) -> torch.Tensor:
    if dist == "uniform":
        return uniform(shape, seed, dtype)
    if dist == "integer":
        return integers(shape, seed, dtype)
    if dist == "normal":
        return normal(shape, seed, std, dtype)
    raise ValueError(f"unknown distribution {dist!r}")


def stored_shape(trans: bool, rows: int, cols: int) -> Tuple[int, int]:
    """Storage shape of an operand whose logical (op) shape is rows x cols."""
    return (cols, rows) if trans else (rows, cols)


@dataclass
class Problem:
    """One GEMM instance: C = alpha*op(A)@op(B) + beta*C_in, CPU tensors."""
    M: int
    N: int
    K: int
    transA: bool
    transB: bool
    dtype: str
    alpha: float
    beta: float
    A: torch.Tensor
    B: torch.Tensor
    C_in: Optional[torch.Tensor]
    name: str = ""


def make_problem(M, N, K, transA=False, transB=False, dtype="f32", dist="uniform", seed=0,
                 alpha=1.0, beta=0.0, std_a=1.0, std_b=1.0, c_fill="uniform",
                 name="") -> Problem:
    """Operands in their stored layouts: A [M,K] (or [K,M] when transA),
    B [K,N] (or [N,K] when transB), C_in [M,N] drawn only when beta != 0
    (c_fill 'uniform' or 'integer')."""
    A = draw(dist, stored_shape(transA, M, K), seed * 3 + 0, dtype, std_a)
    B = draw(dist, stored_shape(transB, K, N), seed * 3 + 1, dtype, std_b)
    C_in = None
    if beta != 0.0:
        C_in = draw(c_fill if dist != "normal" else "uniform", (M, N), seed * 3 + 2, dtype)
    return Problem(M, N, K, bool(transA), bool(transB), dtype, float(alpha), float(beta), A, B,
                   C_in, name)


VARIANTS = {"nn": (False, False), "tn": (True, False), "nt": (False, True), "tt": (True, True)}


# ---------------------------------------------------------------------------
# The workloads: shapes and distributions of the pages' experiments.
# ---------------------------------------------------------------------------
def sgemm_512(integer: bool = False) -> Problem:
    """fp32 nn 512^3, alpha 1 beta 0 (the C-loop post's problem size)."""
    return make_problem(512, 512, 512, dtype="f32", dist="integer" if integer else "uniform",
                        seed=11 if integer else 10, name="f32_nn_512" + ("_int" if integer else ""))


def sgemm_4096() -> Problem:
    """fp32 nn 4096^3, alpha 1 beta 0 (the M5 worklog's problem)."""
    return make_problem(4096, 4096, 4096, dtype="f32", seed=20, name="f32_nn_4096")


def hgemm_square(n: int = 2048, variant: str = "nn", seed: int = 30) -> Problem:
    """fp16 operands / fp32 accumulate / fp16 out, n^3, one of nn/tn/nt."""
    tA, tB = VARIANTS[variant]
    return make_problem(n, n, n, tA, tB, dtype="f16", seed=seed + "nn tn nt tt".split().index(variant),
                        name=f"f16_{variant}_{n}")


@dataclass
class LoraGemm:
    name: str
    variant: str
    M: int
    N: int
    K: int
    beta: float
    a: Tuple[str, float]  # (distribution, std) of the stored A operand
    b: Tuple[str, float]


def lora_step_gemms(T=512, d=2048, F=5632, r=32) -> List[LoraGemm]:
    """The GEMMs of one LoRA MLP-block training step (forward and backward),
    as profiled in "Metal GEMM Kernels for LoRA Training on Apple Silicon",
    section 5: weights stored [out, in] so forward projections are nt, weight
    gradients tn, activation gradients nn.  Activations ~N(0,1), weights
    ~N(0, 0.02^2)."""
    act, w = ("normal", 1.0), ("normal", 0.02)
    g = [
        LoraGemm("fwd_gate", "nt", T, F, d, 0.0, act, w),
        LoraGemm("fwd_up", "nt", T, F, d, 0.0, act, w),
        LoraGemm("fwd_down", "nt", T, d, F, 0.0, act, w),
        LoraGemm("bwd_dS", "nn", T, F, d, 0.0, act, w),
        LoraGemm("bwd_dH_gate", "nn", T, d, F, 0.0, act, w),
        LoraGemm("bwd_dH_up_acc", "nn", T, d, F, 1.0, act, w),
    ]
    for ad in ("gate", "up"):
        g += [
            LoraGemm(f"fwd_{ad}_xA", "nt", T, r, d, 0.0, act, w),
            LoraGemm(f"fwd_{ad}_xAB", "nt", T, F, r, 0.0, act, w),
            LoraGemm(f"bwd_{ad}_dGB", "nn", T, r, F, 0.0, act, w),
            LoraGemm(f"bwd_{ad}_dGBA", "nn", T, d, r, 0.0, act, w),
            LoraGemm(f"bwd_{ad}_dA", "tn", r, d, T, 0.0, act, act),
            LoraGemm(f"bwd_{ad}_dB", "tn", F, r, T, 0.0, act, act),
        ]
    return g


def lora_problem(g: LoraGemm, seed: int, dtype: str = "f16") -> Problem:
    tA, tB = VARIANTS[g.variant]
    A = draw(g.a[0], stored_shape(tA, g.M, g.K), seed * 3 + 0, dtype, g.a[1])
    B = draw(g.b[0], stored_shape(tB, g.K, g.N), seed * 3 + 1, dtype, g.b[1])
    C_in = normal((g.M, g.N), seed * 3 + 2, 1.0, dtype) if g.beta != 0.0 else None
    return Problem(g.M, g.N, g.K, tA, tB, dtype, 1.0, g.beta, A, B, C_in, g.name)


SWEEP_SQUARES = [256, 512, 1024, 2048, 4096, 8192]
SWEEP_ODD = [(4095, 4095, 4095), (1000, 3000, 777), (8192, 32, 8192)]


def sweep_problem(M, N, K, variant, dtype, beta, seed) -> Problem:
    tA, tB = VARIANTS[variant]
    return make_problem(M, N, K, tA, tB, dtype=dtype, seed=seed, beta=beta,
                        alpha=1.0, name=f"{dtype}_{variant}_{M}x{N}x{K}_b{beta}")


# ---------------------------------------------------------------------------
# Strided batches and the attention products ("Metal GEMM Kernels for LoRA
# Training on Apple Silicon", section 8: Q, K, V head-major [H, N, d_h]).
# ---------------------------------------------------------------------------
@dataclass
class BatchedProblem:
    """batch entries of one shape: A [batch, *stored A], B [batch, *stored B],
    C_in [batch, M, N] (None when beta == 0); CPU tensors, contiguous unless a
    test re-lays them out."""
    M: int
    N: int
    K: int
    batch: int
    transA: bool
    transB: bool
    dtype: str
    alpha: float
    beta: float
    A: torch.Tensor
    B: torch.Tensor
    C_in: Optional[torch.Tensor]
    name: str = ""


def batched_problem(M, N, K, batch, variant="nn", dtype="f32", dist="uniform", seed=0, alpha=1.0,
                    beta=0.0, name="") -> BatchedProblem:
    tA, tB = VARIANTS[variant]
    A = draw(dist, (batch,) + stored_shape(tA, M, K), seed * 3 + 0, dtype)
    B = draw(dist, (batch,) + stored_shape(tB, K, N), seed * 3 + 1, dtype)
    C_in = draw(dist, (batch, M, N), seed * 3 + 2, dtype) if beta != 0.0 else None
    return BatchedProblem(M, N, K, batch, tA, tB, dtype, float(alpha), float(beta), A, B, C_in,
                          name or f"{dtype}_{variant}_{batch}x{M}x{N}x{K}")


def causal_probabilities(H, N, seed, dtype="f16") -> torch.Tensor:
    """A synthetic P of the attention forward pass: [H, N, N], row i
    non-negative on columns 0..i, exactly zero above the diagonal (the masked
    half is written as hard zeros), each row scaled to sum to ~1 before
    rounding to the operand type."""
    u = torch.rand((H, N, N), generator=_gen(seed), dtype=torch.float32).double()
    u = torch.tril(u)
    u = u / u.sum(dim=-1, keepdim=True)
    return u.to(DTYPES[dtype])


ATTENTION_PRODUCTS = [
    # (name, variant, left operand, right operand, M, N, K) with n = sequence
    # length and d = head dimension; operands are [H, rows, cols] head-major
    ("S=QK^T", "nt", "Q", "K", "n", "n", "d"),
    ("O=PV", "nn", "P", "V", "n", "d", "n"),
    ("dV=P^T dO", "tn", "P", "dO", "n", "d", "n"),
    ("dP=dO V^T", "nt", "dO", "V", "n", "n", "d"),
    ("dQ=dS K", "nn", "dS", "K", "n", "d", "n"),
    ("dK=dS^T Q", "tn", "dS", "Q", "n", "d", "n"),
]


def attention_tensors(H, n, d, seed, dtype="f16") -> dict:
    """Q, K, V, dO ~ N(0, 1) as [H, n, d]; P a causal row-stochastic [H, n, n];
    dS ~ N(0, 1/n) as [H, n, n] (a stand-in for the softmax backward output,
    which the GEMMs only consume)."""
    t = {nm: normal((H, n, d), seed * 7 + i, 1.0, dtype) for i, nm in enumerate(("Q", "K", "V", "dO"))}
    t["P"] = causal_probabilities(H, n, seed * 7 + 4, dtype)
    t["dS"] = normal((H, n, n), seed * 7 + 5, float(n) ** -0.5, dtype)
    return t
