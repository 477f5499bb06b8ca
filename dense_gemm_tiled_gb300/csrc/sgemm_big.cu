// FP32 SGEMM on the CUDA cores, big tile (the kernel is in sgemm_ffma.cuh):
// 128 x 256 outputs per block, each lane 8 x 16, for problems with enough
// tiles to fill the SMs several times over.
#include "sgemm_ffma.cuh"

namespace gb300 {

cudaError_t launch_sgemm_big(const SgemmArgs& a, LaunchCtx& ctx) {
  return launch_sgemm_t<TileBig, true>(a, ctx);
}

}  // namespace gb300
