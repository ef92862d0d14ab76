// Instantiations of the skinny GEMV / linear kernel for int6 weights.
#include "woq_gemv_launch.cuh"

namespace woq {

cudaError_t launch_gemv_w6(bool fused, int M, const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream) {
  return launch_gemv_bits<6, kern::kDp4a>(fused, M, p, cfg, stream);
}

}  // namespace woq
