// Instantiations of the skinny GEMV / linear for int4 weights, tensor-core consumer, int8 and bf16 prologues.
#include "woq_gemv_launch.cuh"

namespace woq {

cudaError_t launch_w4_mma_plain(int pro, int M, const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream) {
  return launch_gemv_pair<4, kern::kMma, kern::kProInt8, kern::kProBf16>(pro, M, p, cfg, stream);
}

}  // namespace woq
