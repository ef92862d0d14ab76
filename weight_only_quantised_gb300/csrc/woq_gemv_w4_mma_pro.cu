// Instantiations of the skinny linear for int4 weights, tensor-core consumer, RMSNorm and SwiGLU prologues.
#include "woq_gemv_launch.cuh"

namespace woq {

cudaError_t launch_w4_mma_norm(int pro, int M, const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream) {
  return launch_gemv_pair<4, kern::kMma, kern::kProRms, kern::kProSwiglu>(pro, M, p, cfg, stream);
}

}  // namespace woq
