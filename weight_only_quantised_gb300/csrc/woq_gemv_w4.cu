// Instantiations of the skinny GEMV / linear kernel for int4 weights (dp4a consumer).
#include "woq_gemv_launch.cuh"

namespace woq {

cudaError_t launch_gemv_w4(bool fused, int cons, int M, const GemvParams& p, const LaunchConfig& cfg,
                           cudaStream_t stream) {
  if (cons != kern::kDp4a) return launch_gemv_w4_mma(fused, cons, M, p, cfg, stream);
  return launch_gemv_bits<4, kern::kDp4a>(fused, M, p, cfg, stream);
}

}  // namespace woq

#ifdef WOQ_TRACE
// Trace build only: copy the int4 kernel's trace stamps ([16 slots][512 CTAs][64 events]) to the host.
extern "C" __attribute__((visibility("default"))) int woq_trace_read(void* host, size_t bytes) {
  const size_t n = sizeof(woq::g_trace) < bytes ? sizeof(woq::g_trace) : bytes;
  return cudaMemcpyFromSymbol(host, woq::g_trace, n) == cudaSuccess ? 0 : 6;
}
extern "C" __attribute__((visibility("default"))) int woq_trace_clear(void) {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, woq::g_trace) != cudaSuccess) return 6;
  return cudaMemset(ptr, 0, sizeof(woq::g_trace)) == cudaSuccess ? 0 : 6;
}
#endif
