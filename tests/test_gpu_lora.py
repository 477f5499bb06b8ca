"""The GEMMs of one LoRA MLP-block training step (T=512, d=2048, FFN=5632,
rank 32), fp16 storage with fp32 accumulation, as listed in "Metal GEMM Kernels
for LoRA Training on Apple Silicon", section 5 (per-dispatch profile) -- each
against the oracle, then the whole set captured in one CUDA graph and replayed
bit-for-bit."""
import pytest
import torch

from dense_gemm_tiled_gb300 import inputs
from helpers import check_problem

pytestmark = pytest.mark.gpu

GEMMS = inputs.lora_step_gemms()


@pytest.fixture(autouse=True)
def _lib(lib_path, gpu):
    yield


@pytest.mark.parametrize("i", range(len(GEMMS)), ids=[g.name for g in GEMMS])
def test_lora_gemm(i):
    g = GEMMS[i]
    p = inputs.lora_problem(g, seed=500 + i)
    res = check_problem(p)
    assert res["path"] in ("tc", "tc_splitk")


def test_lora_step_cuda_graph_replay_matches_eager():
    from dense_gemm_tiled_gb300 import binding
    probs = [inputs.lora_problem(g, seed=500 + i) for i, g in enumerate(GEMMS)]
    dev = torch.device("cuda:0")
    ops = []
    for p in probs:
        A, B = p.A.to(dev), p.B.to(dev)
        C0 = p.C_in.to(dev) if p.C_in is not None else torch.zeros((p.M, p.N), dtype=torch.float16,
                                                                     device=dev)
        ops.append((A, B, C0, torch.empty_like(C0), p))
    s = torch.cuda.Stream(dev)

    def run_all():
        for A, B, C0, C, p in ops:
            C.copy_(C0)
            binding.gemm(A, B, C, p.transA, p.transB, p.alpha, p.beta, stream=s)

    with torch.cuda.stream(s):
        run_all()  # eager (also the warm-up before capture)
    s.synchronize()
    eager = [C.clone() for _, _, _, C, _ in ops]
    for _, _, _, C, _ in ops:
        C.fill_(float("nan"))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        run_all()
    graph.replay()
    torch.cuda.synchronize()
    for (_, _, _, C, p), ref in zip(ops, eager):
        assert torch.equal(C, ref), p.name
    assert binding.check_device_status() == binding.OK
