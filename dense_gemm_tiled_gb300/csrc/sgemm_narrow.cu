// FP32 SGEMM on the CUDA cores, narrow tile for N <= 32 (the kernel is in
// sgemm_ffma.cuh): 256 x 32 outputs per block, so a rank-32 output keeps every
// lane's columns busy where the general 128 x 128 tile would idle 3/4 of them.
#include "sgemm_ffma.cuh"

namespace gb300 {

cudaError_t launch_sgemm_narrow(const SgemmArgs& a, LaunchCtx& ctx) {
  return launch_sgemm_t<TileNarrow, false>(a, ctx);
}

}  // namespace gb300
