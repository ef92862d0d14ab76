// Instantiations of the skinny linear for int4 weights, dp4a consumer, RMSNorm and SwiGLU prologues.
#include "woq_gemv_launch.cuh"

namespace woq {

cudaError_t launch_w4_dp4a_norm(int pro, int M, const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream) {
  return launch_gemv_pair<4, kern::kDp4a, kern::kProRms, kern::kProSwiglu>(pro, M, p, cfg, stream);
}

}  // namespace woq

#ifdef WOQ_TRACE
// Trace build only: the stamps of this translation unit's kernels (RMSNorm and SwiGLU prologues).
extern "C" __attribute__((visibility("default"))) int woq_trace_read_pro(void* host, size_t bytes) {
  const size_t n = sizeof(woq::g_trace) < bytes ? sizeof(woq::g_trace) : bytes;
  return cudaMemcpyFromSymbol(host, woq::g_trace, n) == cudaSuccess ? 0 : 6;
}
extern "C" __attribute__((visibility("default"))) int woq_trace_clear_pro(void) {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, woq::g_trace) != cudaSuccess) return 6;
  return cudaMemset(ptr, 0, sizeof(woq::g_trace)) == cudaSuccess ? 0 : 6;
}
#endif
