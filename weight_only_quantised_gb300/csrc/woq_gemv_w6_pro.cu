// Instantiations of the skinny linear for int6 weights (dp4a), RMSNorm and SwiGLU prologues.
#include "woq_gemv_launch.cuh"

namespace woq {

cudaError_t launch_w6_norm(int pro, int M, const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream) {
  return launch_gemv_pair<6, kern::kDp4a, kern::kProRms, kern::kProSwiglu>(pro, M, p, cfg, stream);
}

}  // namespace woq
