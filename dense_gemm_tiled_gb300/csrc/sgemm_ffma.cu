// FP32 SGEMM on the CUDA cores, general tile (the kernel is in sgemm_ffma.cuh).
#include "sgemm_ffma.cuh"

namespace gb300 {

cudaError_t launch_sgemm(const SgemmArgs& a, LaunchCtx& ctx) {
  if (a.narrow) return launch_sgemm_narrow(a, ctx);
  return launch_sgemm_t<TileWide, true>(a, ctx);
}

}  // namespace gb300
