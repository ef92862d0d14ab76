// Instantiations of the skinny GEMV / linear kernel for int4 weights (tensor-core consumer).
#include "woq_gemv_launch.cuh"

namespace woq {

cudaError_t launch_gemv_w4_mma(bool fused, int cons, int M, const GemvParams& p, const LaunchConfig& cfg,
                               cudaStream_t stream) {
  (void)cons;
  return launch_gemv_bits<4, kern::kMma>(fused, M, p, cfg, stream);
}

}  // namespace woq
