// bf16 instantiation of the tcgen05 GEMM (hgemm_tcgen05.cuh): bfloat16
// operands and output, fp32 accumulation.  bfloat16 is listed in the operand
// type table of "Metal GEMM Kernels for LoRA Training on Apple Silicon",
// section 1 (emulated on that GPU); kind::f16 tensor-core MMAs take it natively
// at the fp16 rate.
#include "hgemm_tcgen05.cuh"

namespace gb300 {

cudaError_t launch_hgemm_bf16(const HgemmArgs& a, LaunchCtx& ctx) {
  return launch_hgemm_t<__nv_bfloat16>(a, ctx);
}

}  // namespace gb300
