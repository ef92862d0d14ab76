// Launch helpers for the GEMV / linear kernel (programmatic dependent launch).
#pragma once

#include <atomic>

#include "woq_gemv.cuh"
#include "woq_internal.h"

namespace woq {

template <int BITS, int M, int PRO, int CONS>
cudaError_t launch_gemv_instance(const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream) {
  auto kernel = kern::gemv_kernel<BITS, M, PRO, CONS>;
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

template <int BITS, int PRO, int CONS>
cudaError_t launch_gemv_m(int M, const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream) {
  switch (M) {
    case 1: return launch_gemv_instance<BITS, 1, PRO, CONS>(p, cfg, stream);
    case 2: return launch_gemv_instance<BITS, 2, PRO, CONS>(p, cfg, stream);
    case 3: return launch_gemv_instance<BITS, 3, PRO, CONS>(p, cfg, stream);
    case 4: return launch_gemv_instance<BITS, 4, PRO, CONS>(p, cfg, stream);
    default: break;
  }
  if constexpr (CONS == kern::kMma) {  // five to eight rows: tensor-core consumer only
    switch (M) {
      case 5: return launch_gemv_instance<BITS, 5, PRO, CONS>(p, cfg, stream);
      case 6: return launch_gemv_instance<BITS, 6, PRO, CONS>(p, cfg, stream);
      case 7: return launch_gemv_instance<BITS, 7, PRO, CONS>(p, cfg, stream);
      case 8: return launch_gemv_instance<BITS, 8, PRO, CONS>(p, cfg, stream);
      default: break;
    }
  }
  return cudaErrorInvalidValue;
}

// Instances of two prologues (pro = PRO_A or PRO_B) for one (BITS, consumer) pair.
template <int BITS, int CONS, int PRO_A, int PRO_B>
cudaError_t launch_gemv_pair(int pro, int M, const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream) {
  if (pro == PRO_A) return launch_gemv_m<BITS, PRO_A, CONS>(M, p, cfg, stream);
  if (pro == PRO_B) return launch_gemv_m<BITS, PRO_B, CONS>(M, p, cfg, stream);
  return cudaErrorInvalidValue;
}

// One translation unit each, so that the instances compile in parallel:
//   woq_gemv_w4.cu (int4 dp4a: int8 and bf16 prologues, and the dispatcher below),
//   woq_gemv_w4_pro.cu (int4 dp4a: RMSNorm and SwiGLU), woq_gemv_w4_mma.cu and
//   woq_gemv_w4_mma_pro.cu (the same for the tensor-core consumer), woq_gemv_w6.cu and
//   woq_gemv_w6_pro.cu (int6).
cudaError_t launch_w4_dp4a_plain(int pro, int M, const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream);
cudaError_t launch_w4_dp4a_norm(int pro, int M, const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream);
cudaError_t launch_w4_mma_plain(int pro, int M, const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream);
cudaError_t launch_w4_mma_norm(int pro, int M, const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream);
cudaError_t launch_w6_plain(int pro, int M, const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream);
cudaError_t launch_w6_norm(int pro, int M, const GemvParams& p, const LaunchConfig& cfg, cudaStream_t stream);

// bits 4 or 6, pro a kern::Prologue, cons a kern::Consumer (int6: dp4a only)
cudaError_t launch_gemv_any(int bits, int pro, int cons, int M, const GemvParams& p, const LaunchConfig& cfg,
                            cudaStream_t stream);

}  // namespace woq
