// Instantiations of the skinny GEMV / linear kernel for int4 weights (dp4a consumer).
#include "woq_gemv_launch.cuh"

namespace woq {

cudaError_t launch_w4_dp4a_plain(int pro, int M, const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream) {
  return launch_gemv_pair<4, kern::kDp4a, kern::kProInt8, kern::kProBf16>(pro, M, p, cfg, stream);
}

cudaError_t launch_gemv_any(int bits, int pro, int cons, int M, const GemvParams& p, const LaunchConfig& cfg,
                            cudaStream_t stream) {
  const bool plain = pro == kern::kProInt8 || pro == kern::kProBf16;
  if (bits == 6) return plain ? launch_w6_plain(pro, M, p, cfg, stream) : launch_w6_norm(pro, M, p, cfg, stream);
  if (cons == kern::kMma)
    return plain ? launch_w4_mma_plain(pro, M, p, cfg, stream) : launch_w4_mma_norm(pro, M, p, cfg, stream);
  return plain ? launch_w4_dp4a_plain(pro, M, p, cfg, stream) : launch_w4_dp4a_norm(pro, M, p, cfg, stream);
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
