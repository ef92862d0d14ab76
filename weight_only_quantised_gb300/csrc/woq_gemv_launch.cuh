// Launch helpers for the GEMV / linear kernel (programmatic dependent launch).
#pragma once

#include <atomic>

#include "woq_gemv.cuh"
#include "woq_internal.h"

namespace woq {

template <int BITS, int M, bool FUSED, int CONS>
cudaError_t launch_gemv_instance(const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream) {
  auto kernel = kern::gemv_kernel<BITS, M, FUSED, CONS>;
  // raise the kernel's dynamic shared-memory limit once per device
  static std::atomic<unsigned long long> configured{0};
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (device & 63);
  if (!(configured.load(std::memory_order_relaxed) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dynamic_smem());
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)cfg.ctas, 1, 1);
  lc.blockDim = dim3((unsigned)kThreads, 1, 1);
  lc.dynamicSmemBytes = (size_t)cfg.smem_bytes;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kernel, p);
}

template <int BITS, bool FUSED, int CONS>
cudaError_t launch_gemv_m(int M, const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream) {
  switch (M) {
    case 1: return launch_gemv_instance<BITS, 1, FUSED, CONS>(p, cfg, stream);
    case 2: return launch_gemv_instance<BITS, 2, FUSED, CONS>(p, cfg, stream);
    case 3: return launch_gemv_instance<BITS, 3, FUSED, CONS>(p, cfg, stream);
    case 4: return launch_gemv_instance<BITS, 4, FUSED, CONS>(p, cfg, stream);
    default: break;
  }
  if constexpr (CONS == kern::kMma) {  // five to eight rows: tensor-core consumer only
    switch (M) {
      case 5: return launch_gemv_instance<BITS, 5, FUSED, CONS>(p, cfg, stream);
      case 6: return launch_gemv_instance<BITS, 6, FUSED, CONS>(p, cfg, stream);
      case 7: return launch_gemv_instance<BITS, 7, FUSED, CONS>(p, cfg, stream);
      case 8: return launch_gemv_instance<BITS, 8, FUSED, CONS>(p, cfg, stream);
      default: break;
    }
  }
  return cudaErrorInvalidValue;
}

template <int BITS, int CONS>
cudaError_t launch_gemv_bits(bool fused, int M, const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream) {
  return fused ? launch_gemv_m<BITS, true, CONS>(M, p, cfg, stream) : launch_gemv_m<BITS, false, CONS>(M, p, cfg, stream);
}

// cons: kern::Consumer of the launch (int4 only; int6 is always dp4a)
cudaError_t launch_gemv_w4(bool fused, int cons, int M, const GemvParams& p, const LaunchConfig& cfg,
                           cudaStream_t stream);
cudaError_t launch_gemv_w4_mma(bool fused, int cons, int M, const GemvParams& p, const LaunchConfig& cfg,
                               cudaStream_t stream);
cudaError_t launch_gemv_w6(bool fused, int M, const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream);

}  // namespace woq
