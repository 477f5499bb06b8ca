// FP32 SGEMM on the CUDA cores, general tile (the kernel is in sgemm_ffma.cuh).
#include "sgemm_ffma.cuh"

namespace gb300 {

cudaError_t launch_sgemm(const SgemmArgs& a, LaunchCtx& ctx) {
  if (a.tile == SG_TILE_NARROW) return launch_sgemm_narrow(a, ctx);
  if (a.tile == SG_TILE_BIG) return launch_sgemm_big(a, ctx);
  if (a.tile == SG_TILE_HALF) return launch_sgemm_half(a, ctx);
  return launch_sgemm_t<TileWide, true>(a, ctx);
}

}  // namespace gb300
