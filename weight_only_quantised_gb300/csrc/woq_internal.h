// Internal declarations shared by the library's translation units.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime.h>

namespace woq {

void write_header(void* dst, int bits, int N, int K);
bool header_matches(const void* src, int bits, int N, int K);

// Launch configuration of one GEMV / linear launch (chosen by the launch table).
struct LaunchConfig {
  int ctas;             // grid size (CTAs); each CTA streams an equal share of the blocks
  int stages;           // ring stages of kStageBlocks blocks each
  int smem_bytes;       // dynamic shared memory per CTA
  int prefetch_stages;  // stages kept in flight into L2 beyond the ring
  int consumer;         // kern::Consumer (dp4a or tensor-core MMA)
};

// Workspace layout: [status word + pad: 256 B][tagged partial sums: ctas x 2 x M x 128 x 8 B]
struct WorkspaceLayout {
  size_t parts_offset;  // split-tile partial sums
  size_t h_offset;      // SwiGLU prologue scratch rows (bf16 [M][K]); no zeroing needed
  size_t total;
};

constexpr int kConsumerWarps = 8;
constexpr int kStageBlocks = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 8;

int sm_count();                       // SMs of the current device (cached per device)
int max_dynamic_smem();               // opt-in shared memory per block of the current device
int choose_consumer(int bits, int M);  // kern::Consumer the launch table picks for (bits, M)
int smem_bytes_for(int bits, int M, int K, bool fused, int stages);
// resident_grid: the launch has a grid-wide step (the SwiGLU prologue), so its CTAs must all be
// resident at once: at most one per SM, whatever the tuning override says
LaunchConfig choose_config(int bits, int M, int N, int K, bool fused, bool resident_grid = false);
// The same choice for a device with sms SMs and smem_max bytes of opt-in shared memory per block
// (ctas == 0 when nothing fits).
LaunchConfig choose_config_for(int sms, int smem_max, int bits, int M, int N, int K, bool fused, bool resident_grid);
WorkspaceLayout workspace_layout(int M, int N, int K, int ctas);

// Kernel launchers (woq_gemv.cu); return a cudaError_t.
cudaError_t launch_gemv(int bits, bool fused, int M, int N, int K, const void* wpacked, const void* x_bf16,
                        const int8_t* q, const float* ascale, float* y, void* ws, const LaunchConfig& cfg,
                        const WorkspaceLayout& wl, cudaStream_t stream);
cudaError_t launch_act_quant(const void* x_bf16, int M, int K, int8_t* q, float* ascale, cudaStream_t stream);
// pro: kern::kProRms (x bf16 [M][K], gamma bf16 [K]) or kern::kProSwiglu (x fp32 [M][2K])
cudaError_t launch_pro_act_quant(int pro, const void* x, const uint16_t* gamma, float eps, int M, int K, int8_t* q,
                                 float* ascale, cudaStream_t stream);
cudaError_t launch_group_dots(int bits, const void* wpacked, const int8_t* q, int M, int N, int K, int32_t* dots,
                              cudaStream_t stream);
cudaError_t launch_pack_device(int bits, const uint8_t* q, const uint16_t* scales, int N, int K, void* dst,
                               cudaStream_t stream);
// in-place relayout; *too_large = 1 (and nothing launched) if the staging does not fit.  wait_ns bounds
// the waits on other CTAs; fault_cta >= 0 injects a CTA that never arrives (tests of that bound).
cudaError_t launch_relayout(int bits, void* buf, int N, int K, int* too_large, cudaStream_t stream,
                            unsigned long long wait_ns, int fault_cta);

}  // namespace woq
