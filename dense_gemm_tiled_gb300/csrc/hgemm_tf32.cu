// Opt-in TF32 GEMM: the tcgen05 kernel of hgemm_tcgen05.cuh instantiated for
// fp32 operands and output with kind::tf32 MMAs.  The tensor core uses the TF32
// part of each fp32 operand (8 exponent bits, 10 fraction bits) and accumulates
// in fp32: a reduced-precision alternative to the FFMA SGEMM, offered only on
// request (the counterpart of the relaxed-precision switch that "Optimizing GEMM
// on Apple's M5 from scratch, Part 2" leaves off, section "Precision, Timing,
// and the Neural Accelerators").  Operands are K-major (A [M, K], B [N, K]);
// the dispatcher packs other layouts first.
#include "hgemm_tcgen05.cuh"

namespace gb300 {

cudaError_t launch_hgemm_tf32(const HgemmArgs& a, LaunchCtx& ctx) {
  return launch_hgemm_t<float>(a, ctx);
}

}  // namespace gb300
