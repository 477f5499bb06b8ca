// FP32 SGEMM on the CUDA cores, half tile (the kernel is in sgemm_ffma.cuh):
// 128 x 64 outputs per block, two blocks per SM, for grids of 128 x 128 tiles
// that would leave SMs idle.
#include "sgemm_ffma.cuh"

namespace gb300 {

cudaError_t launch_sgemm_half(const SgemmArgs& a, LaunchCtx& ctx) {
  return launch_sgemm_t<TileHalf, true>(a, ctx);
}

}  // namespace gb300
