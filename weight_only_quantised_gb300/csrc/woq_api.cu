// C ABI of the skinny linear: argument validation, the per-shape launch table
// and the device entry points.  Everything here is host code; every step of
// the computation runs in the kernels of woq_gemv.cuh and woq_small_kernels.cu.
#include <atomic>
#include <mutex>

#include "woq.h"
#include "woq_gemv_launch.cuh"
#include "woq_internal.h"
#include "woq_layout.h"

namespace woq {

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_max_smem[kMaxDevices];
std::atomic<int> g_override_cps{0};
std::atomic<int> g_override_stages{0};
std::atomic<int> g_override_prefetch_kb{-1};
std::atomic<int> g_override_path{0};  // 0: table, else 1 + kern::Consumer
std::atomic<int> g_launch_counter{0};  // numbers GEMV launches (trace builds key their stamps by it)
// woq_tune_fault: a fault to inject (0 none, 1 split-tile publish, 2 SwiGLU arrival, 3 relayout
// barrier arrival) by one CTA, and the bound of the waits it makes run out (0 = the default)
std::atomic<int> g_fault_kind{0};
std::atomic<int> g_fault_cta{0};
std::atomic<long long> g_wait_ns{0};
uint64_t wait_bound_ns() {
  const long long v = g_wait_ns.load(std::memory_order_relaxed);
  return v > 0 ? (uint64_t)v : dev::kWaitLimitNs;
}

// A failed CUDA call: remembered for woq_last_cuda_error (per thread) and cleared from the
// runtime's error state, so that it does not surface again in the caller's next call.
thread_local int t_last_cuda_error = 0;
int cuda_result(cudaError_t e) {
  if (e == cudaSuccess) return WOQ_OK;
  t_last_cuda_error = (int)e;
  (void)cudaGetLastError();
  return WOQ_ERR_CUDA;
}

int current_device() {
  int d = 0;
  if (const cudaError_t e = cudaGetDevice(&d); e != cudaSuccess) {
    cuda_result(e);
    return -1;
  }
  return d;
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

int sm_count() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return 0;
  int v = g_sm_count[d].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) return 0;
    g_sm_count[d].store(v, std::memory_order_relaxed);
  }
  return v;
}

int max_dynamic_smem() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return 0;
  int v = g_max_smem[d].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, d) != cudaSuccess) return 0;
    g_max_smem[d].store(v, std::memory_order_relaxed);
  }
  return v;
}

// [barriers, flags, scratch: 1024][reduction buffer][activations][ring]
// activations: bf16 x quantised in place (fused, 2 M K bytes) or int8 q (M rows); kernels
// with tensor-core warps read q rows padded to K + 16 bytes (conflict-free fragment loads).
// In the fused entry q needs only the first M (K or K + 16) bytes once the prologue is
// done, and the reduction buffer is first written after it, so when the bf16 tail is
// large enough the reduction buffer lives there: [1024][activations (q + reduction)][ring].
static int red_bytes(int M) { return kStageBlocks * M * kTileRows * 4; }
static constexpr int kMiscBytes = 1024;  // barriers, flags, row scales and scratch (see the kernel)
static int act_stride(int K, int cons) { return cons != kern::kDp4a ? K + 16 : K; }
static int act_bytes(int M, int K, bool fused, int cons) { return fused ? 2 * M * K : M * act_stride(K, cons); }
static int q_end(int M, int K, int cons) { return (int)align_up((size_t)M * act_stride(K, cons), 16); }
static bool red_in_act(int M, int K, bool fused, int cons) {
  return fused && q_end(M, K, cons) + red_bytes(M) <= act_bytes(M, K, fused, cons);
}
static int act_offset(int M, int K, bool fused, int cons) {
  return kMiscBytes + (red_in_act(M, K, fused, cons) ? 0 : red_bytes(M));
}
static int red_offset(int M, int K, bool fused, int cons) {
  return red_in_act(M, K, fused, cons) ? act_offset(M, K, fused, cons) + q_end(M, K, cons) : kMiscBytes;
}
static int ring_offset(int M, int K, bool fused, int cons) {
  return (int)align_up((size_t)act_offset(M, K, fused, cons) + (size_t)act_bytes(M, K, fused, cons), 128);
}

// Consumer of the int4 kernels (kern::Consumer).  dp4a for M <= 4: on this part the f16
// MMA (mma.sync, fp32 accumulate) costs about what dp4a costs at M = 4 and more below it,
// and the two contend when mixed in one SM sub-partition.  The MMA's cost does not grow with
// M, so it takes M = 5 .. 8 (no dp4a kernel exists there); for M <= 4 woq_tune_path can
// select it.  int6 is always dp4a (M <= 4).
int choose_consumer(int bits, int M) {
  if (bits != 4) return kern::kDp4a;
  if (M > kMaxMDp4a) return kern::kMma;
  const int path = g_override_path.load(std::memory_order_relaxed);
  if (path > 0) return path - 1;
  return kern::kDp4a;
}

static int max_m_for(int bits) { return bits == 4 ? kMaxM : kMaxMDp4a; }

int smem_bytes_for(int bits, int M, int K, bool fused, int stages) {
  return ring_offset(M, K, fused, choose_consumer(bits, M)) + stages * kStageBlocks * block_bytes(bits);
}

// Shared memory a launch's ring and activations may take when the tuning override runs two CTAs
// per SM.  By default the kernel runs one CTA per SM (nine warps of 100 or more registers: the
// 16,384-register file of a sub-partition then holds at most four, so a second CTA never fits),
// and the next launch's CTA takes over an SM as soon as this launch's CTA there exits.
static constexpr int kRingBudget = (233472 - 2 * 1024) / 2;

LaunchConfig choose_config(int bits, int M, int N, int K, bool fused, bool resident_grid) {
  return choose_config_for(sm_count(), max_dynamic_smem(), bits, M, N, K, fused, resident_grid);
}

LaunchConfig choose_config_for(int sms, int smem_max, int bits, int M, int N, int K, bool fused, bool resident_grid) {
  LaunchConfig cfg = {0, 0, 0, 0, 0};
  if (sms <= 0 || smem_max <= 0) return cfg;
  const long long T = (N + kTileRows - 1) / kTileRows;
  const long long G = K / kGroup;
  const long long NB = T * G;
  if (NB <= 0) return cfg;
  int cps = g_override_cps.load(std::memory_order_relaxed);
  // one CTA per SM is always resident (a CTA fits an SM alone or the launch fails); a second
  // one never is (the kernels use 100 or more registers), so a grid-wide step would wait for a
  // wave that cannot start
  if (cps <= 0 || resident_grid) cps = 1;
  const int ring_budget = kRingBudget < smem_max ? kRingBudget : smem_max;
  int stages = g_override_stages.load(std::memory_order_relaxed);
  if (stages > 0) {
    const int budget = cps == 1 ? smem_max : ring_budget;
    while (stages >= 2 && smem_bytes_for(bits, M, K, fused, stages) > budget) --stages;
  } else {
    // three stages wherever they fit the device's shared memory (two rows, and five or more,
    // four), else the largest ring that fits.  27B step: three stages everywhere against up to
    // four within half the shared memory (which left the down projection and every M = 4 launch
    // two): M = 1 2.222 -> 2.193 ms, M = 3 2.975 -> 2.920, M = 4 3.388 -> 3.362; at M = 2 three and
    // four stages are even (2.534 ms) and two lose (2.616); four at M = 1 lose (2.241).
    stages = (M == 2 || M >= 5) ? 4 : 3;
    while (stages >= 2 && smem_bytes_for(bits, M, K, fused, stages) > smem_max) --stages;
  }
  if (stages < 2) return cfg;
  const int stage_bytes = kStageBlocks * block_bytes(bits);
  // L2 prefetch window beyond the ring: one stage by default.  A deeper window puts the
  // next launch's whole share in the memory queues at once, and the small critical-path
  // reads of the running launch (activations, split-tile partials) then wait behind it.
  // One row and a large matrix (at least 5000 blocks: the 27B gate_up, down and LM head) take a
  // two-stage window: the next launch's stream then covers more of this launch's prologue
  // (27B step at M = 1: 2.360 -> 2.340 ms; at M = 4 the same rule cost 0.7 %).
  int pf_kb = g_override_prefetch_kb.load(std::memory_order_relaxed);
  if (pf_kb < 0) pf_kb = (M == 1 && NB >= 5000 ? 2 : 1) * stage_bytes / 1024;
  // at least one stage (kStageBlocks blocks) of work per CTA
  long long ctas = (long long)sms * cps;
  const long long by_work = (NB + kStageBlocks - 1) / kStageBlocks;
  if (ctas > by_work) ctas = by_work;
  if (ctas < 1) ctas = 1;
  cfg.ctas = (int)ctas;
  cfg.stages = stages;
  cfg.smem_bytes = smem_bytes_for(bits, M, K, fused, stages);
  cfg.prefetch_stages = (int)(((long long)pf_kb * 1024 + stage_bytes - 1) / stage_bytes);
  cfg.consumer = choose_consumer(bits, M);
  return cfg;
}

// workspace: [0] status word, [64, 128) grid-barrier and row words of the SwiGLU prologue,
// [256, ...) split-tile partial sums
static constexpr size_t kSyncOffset = 64;

WorkspaceLayout workspace_layout(int M, int N, int K, int ctas) {
  (void)N;
  WorkspaceLayout wl;
  wl.parts_offset = 256;
  wl.h_offset = align_up(wl.parts_offset + (size_t)ctas * 2 * (size_t)M * kTileRows * 8, 256);
  wl.total = wl.h_offset + (size_t)M * (size_t)K * 2;
  return wl;
}

// workspace is sized for the largest grid the table or an override may pick
static int max_ctas_for_workspace() { return 2 * sm_count(); }

// Bytes of workspace a launch reads or writes: the status and synchronisation words and the
// split-tile partials, plus the scratch rows for the SwiGLU prologue (the only one using them).
static size_t workspace_need(int pro, const WorkspaceLayout& wl) {
  return pro == kern::kProSwiglu ? wl.total : wl.h_offset;
}

}  // namespace woq

using namespace woq;

extern "C" {

int woq_version(void) { return 200; }

int woq_max_m(void) { return kMaxM; }

const char* woq_status_string(int status) {
  switch (status) {
    case WOQ_OK: return "ok";
    case WOQ_ERR_NULL: return "a required pointer is NULL";
    case WOQ_ERR_ALIGN: return "a device pointer is not suitably aligned";
    case WOQ_ERR_SHAPE: return "M, N, K or bits outside the supported range";
    case WOQ_ERR_WORKSPACE: return "workspace smaller than woq_workspace_bytes()";
    case WOQ_ERR_LAYOUT: return "packed buffer size or header does not match (bits, N, K)";
    case WOQ_ERR_CUDA: return "a CUDA runtime call failed";
    case WOQ_ERR_DEVICE: return "a kernel reported an error in the workspace status word";
    default: return "unknown status";
  }
}

int woq_last_cuda_error(void) { return t_last_cuda_error; }

const char* woq_cuda_error_name(int code) { return cudaGetErrorName((cudaError_t)code); }

int woq_tune_override(int ctas_per_sm, int stages, int prefetch_kb) {
  if (ctas_per_sm < 0 || ctas_per_sm > 2 || stages < 0 || stages == 1 || stages > kMaxStages || prefetch_kb < -1 ||
      prefetch_kb > 65536)
    return WOQ_ERR_SHAPE;
  g_override_cps.store(ctas_per_sm);
  g_override_stages.store(stages);
  g_override_prefetch_kb.store(prefetch_kb);
  return WOQ_OK;
}

int woq_tune_fault(int kind, int cta, int wait_limit_us) {
  if (kind < 0 || kind > 3 || cta < 0 || wait_limit_us < 0 || wait_limit_us > 2000000) return WOQ_ERR_SHAPE;
  g_fault_kind.store(kind);
  g_fault_cta.store(cta);
  g_wait_ns.store((long long)wait_limit_us * 1000);
  return WOQ_OK;
}

int woq_tune_path(int path) {
  if (path < 0 || path > 2) return WOQ_ERR_SHAPE;
  g_override_path.store(path);
  return WOQ_OK;
}

int woq_plan_launch(int bits, int M, int N, int K, int entry, int sms, int smem_max, woq_launch_plan* out) {
  if (!out) return WOQ_ERR_NULL;
  if ((bits != 4 && bits != 6) || M < 1 || M > max_m_for(bits) || N < 1 || K < kGroup || K % kGroup ||
      (long)M * K > kMaxMK || entry < 0 || entry > 2 || sms < 0 || smem_max < 0)
    return WOQ_ERR_SHAPE;
  if (sms == 0) sms = sm_count();
  if (smem_max == 0) smem_max = max_dynamic_smem();
  if (sms <= 0 || smem_max <= 0) return WOQ_ERR_CUDA;
  const LaunchConfig cfg = choose_config_for(sms, smem_max, bits, M, N, K, entry != 0, entry == 2);
  if (cfg.ctas <= 0) return WOQ_ERR_SHAPE;
  const unsigned long long nb = (unsigned long long)((N + kTileRows - 1) / kTileRows) * (unsigned long long)(K / kGroup);
  if ((nb + 1) * (unsigned long long)(cfg.ctas + 1) >= (1ull << 32)) return WOQ_ERR_SHAPE;
  out->ctas = cfg.ctas;
  out->stages = cfg.stages;
  out->prefetch_stages = cfg.prefetch_stages;
  out->smem_bytes = cfg.smem_bytes;
  out->consumer = cfg.consumer;
  return WOQ_OK;
}

int woq_max_k(int bits, int M, int fused) {
  if ((bits != 4 && bits != 6) || M < 1 || M > max_m_for(bits)) return 0;
  const int smem_max = max_dynamic_smem();
  if (smem_max <= 0) return 0;
  int K = (int)(kMaxMK / M) / kGroup * kGroup;
  while (K > 0 && smem_bytes_for(bits, M, K, fused != 0, 2) > smem_max) K -= kGroup;
  return K;
}

size_t woq_workspace_bytes(int bits, int M, int N, int K) {
  if ((bits != 4 && bits != 6) || M < 0 || M > max_m_for(bits) || N < 0 || K < 0 || K % kGroup) return 0;
  if (M == 0 || N == 0 || K == 0) return 256;  // empty shapes launch nothing
  const int c = max_ctas_for_workspace();
  if (c <= 0) return 0;
  return workspace_layout(M, N, K, c).total;
}

int woq_workspace_init(void* ws_dev, size_t ws_bytes, woq_stream_t stream) {
  if (!ws_dev) return WOQ_ERR_NULL;
  if (!aligned(ws_dev, 16)) return WOQ_ERR_ALIGN;
  return cuda_result(cudaMemsetAsync(ws_dev, 0, ws_bytes, (cudaStream_t)stream));
}

int woq_read_status(void* ws_dev, size_t ws_bytes, int clear, uint32_t* status_out, woq_stream_t stream) {
  if (!ws_dev || !status_out) return WOQ_ERR_NULL;
  if (ws_bytes < 4) return WOQ_ERR_WORKSPACE;
  uint32_t v = 0;
  cudaStream_t s = (cudaStream_t)stream;
  if (const cudaError_t e_ = cudaMemcpyAsync(&v, ws_dev, 4, cudaMemcpyDeviceToHost, s); e_ != cudaSuccess)
    return cuda_result(e_);
  if (const cudaError_t e_ = cudaStreamSynchronize(s); e_ != cudaSuccess) return cuda_result(e_);
  if (clear && v) {
    if (const cudaError_t e_ = cudaMemsetAsync(ws_dev, 0, 4, s); e_ != cudaSuccess) return cuda_result(e_);
    if (const cudaError_t e_ = cudaStreamSynchronize(s); e_ != cudaSuccess) return cuda_result(e_);
  }
  *status_out = v;
  return WOQ_OK;
}

int woq_pack_device(int bits, const uint8_t* q_dev, const uint16_t* scales_dev, int N, int K, void* dst_dev,
                    size_t dst_bytes, woq_stream_t stream) {
  const size_t need = packed_bytes(bits, N, K);
  if (need == 0) return WOQ_ERR_SHAPE;
  if (!dst_dev || ((!q_dev || !scales_dev) && (size_t)N * (size_t)K > 0)) return WOQ_ERR_NULL;
  if (!aligned(dst_dev, 16) || !aligned(q_dev, 16) || !aligned(scales_dev, 2)) return WOQ_ERR_ALIGN;
  if (dst_bytes < need) return WOQ_ERR_LAYOUT;
  return cuda_result(launch_pack_device(bits, q_dev, scales_dev, N, K, dst_dev, (cudaStream_t)stream));
}

int woq_relayout_inplace(int bits, void* buf, size_t buf_bytes, int N, int K, woq_stream_t stream) {
  const size_t need = packed_bytes(bits, N, K);
  if (need == 0) return WOQ_ERR_SHAPE;
  if (!buf) return WOQ_ERR_NULL;
  if (!aligned(buf, 16)) return WOQ_ERR_ALIGN;
  if (buf_bytes < need) return WOQ_ERR_LAYOUT;
  if (N == 0 || K == 0) {  // nothing to move: the header alone
    alignas(16) uint8_t h[kHeaderBytes];
    write_header(h, bits, N, K);
    cudaError_t e = cudaMemcpyAsync(buf, h, kHeaderBytes, cudaMemcpyHostToDevice, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    return cuda_result(e);
  }
  int too_large = 0;
  const int fault_cta = g_fault_kind.load(std::memory_order_relaxed) == 3 ? g_fault_cta.load(std::memory_order_relaxed) : -1;
  cudaError_t e = launch_relayout(bits, buf, N, K, &too_large, (cudaStream_t)stream, wait_bound_ns(), fault_cta);
  if (too_large) return WOQ_ERR_SHAPE;
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  uint32_t head[4] = {0u, 0u, 0u, 0u};
  if (e == cudaSuccess) e = cudaMemcpy(head, buf, sizeof(head), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_result(e);
  return head[0] == kMagic ? WOQ_OK : WOQ_ERR_DEVICE;
}

int woq_act_quant_int8(const void* x_bf16, int M, int K, int8_t* q, float* ascale, woq_stream_t stream) {
  if (M < 0 || M > kMaxM || K < 0) return WOQ_ERR_SHAPE;
  if (M == 0) return WOQ_OK;
  if (!ascale || (K > 0 && (!x_bf16 || !q))) return WOQ_ERR_NULL;
  if (!aligned(x_bf16, 16) || !aligned(q, 16) || !aligned(ascale, 4)) return WOQ_ERR_ALIGN;
  return cuda_result(launch_act_quant(x_bf16, M, K, q, ascale, (cudaStream_t)stream));
}

int woq_rmsnorm_act_quant_int8(const void* x_bf16, const void* gamma_bf16, float eps, int M, int K, int8_t* q,
                               float* ascale, woq_stream_t stream) {
  if (M < 0 || M > kMaxM || K < 0 || K % 8 || (size_t)K * 2 > (size_t)max_dynamic_smem()) return WOQ_ERR_SHAPE;
  if (!(eps >= 0.0f && eps <= 3.4028234e38f)) return WOQ_ERR_SHAPE;
  if (M == 0) return WOQ_OK;
  if (!ascale || (K > 0 && (!x_bf16 || !q || !gamma_bf16))) return WOQ_ERR_NULL;
  if (!aligned(x_bf16, 16) || !aligned(gamma_bf16, 16) || !aligned(q, 16) || !aligned(ascale, 4)) return WOQ_ERR_ALIGN;
  return cuda_result(launch_pro_act_quant(kern::kProRms, x_bf16, static_cast<const uint16_t*>(gamma_bf16), eps, M, K, q,
                                          ascale, (cudaStream_t)stream));
}

int woq_swiglu_act_quant_int8(const float* gate_up, int M, int K, int8_t* q, float* ascale, woq_stream_t stream) {
  if (M < 0 || M > kMaxM || K < 0 || K % 8 || (size_t)K * 2 > (size_t)max_dynamic_smem()) return WOQ_ERR_SHAPE;
  if (M == 0) return WOQ_OK;
  if (!ascale || (K > 0 && (!gate_up || !q))) return WOQ_ERR_NULL;
  if (!aligned(gate_up, 16) || !aligned(q, 16) || !aligned(ascale, 4)) return WOQ_ERR_ALIGN;
  return cuda_result(launch_pro_act_quant(kern::kProSwiglu, gate_up, nullptr, 0.0f, M, K, q, ascale, (cudaStream_t)stream));
}

// The next-linear hint of this thread (woq_prefetch_next), consumed by its next GEMV / linear call.
struct NextHint {
  const void* w;
  int bits, N, K, kb;
};
static thread_local NextHint t_next = {nullptr, 0, 0, 0, 0};
static constexpr int kPrefetchNextKb = 64;  // default per-CTA prefetch of the next linear (27B step: 32 - 96 KiB swept)

// Fill the next-linear prefetch fields of p from a hint (none if the hint is empty or its
// partition does not fit the 32-bit math); the next launch is planned like this one.
static void plan_next_prefetch(GemvParams& p, const NextHint& h, int M, bool fused) {
  p.nx_w = nullptr;
  p.nx_NB = p.nx_C = p.nx_bb = p.nx_blocks = 0;
  p.nx_div_c = FastDiv::make(1u);
  p.nx_div_g = FastDiv::make(1u);
  if (!h.w || h.N <= 0 || h.K <= 0) return;
  const int mm = M <= max_m_for(h.bits) ? M : max_m_for(h.bits);
  const LaunchConfig nc = choose_config(h.bits, mm, h.N, h.K, fused, false);
  if (nc.ctas <= 0) return;
  const unsigned long long T = (unsigned long long)((h.N + kTileRows - 1) / kTileRows), G = (unsigned long long)(h.K / kGroup);
  const unsigned long long nb = T * G;
  if ((nb + 1) * (unsigned long long)(nc.ctas + 1) >= (1ull << 32)) return;
  const uint32_t bb = (uint32_t)block_bytes(h.bits);
  const uint32_t blocks = (uint32_t)(((unsigned long long)(h.kb > 0 ? h.kb : kPrefetchNextKb) * 1024ull) / bb);
  if (blocks == 0) return;
  p.nx_w = static_cast<const uint8_t*>(h.w);
  p.nx_NB = (uint32_t)nb;
  p.nx_C = (uint32_t)nc.ctas;
  p.nx_bb = bb;
  p.nx_blocks = blocks;
  p.nx_div_c = FastDiv::make((uint32_t)nc.ctas);
  p.nx_div_g = FastDiv::make((uint32_t)G);
}

// pro: kern::Prologue.  x: bf16 [M][K] (bf16, RMSNorm) or fp32 [M][2K] (SwiGLU).
static int run_gemv(int bits, int pro, const void* wpacked, size_t wpacked_bytes, const void* x, const int8_t* q,
                    const float* ascale, const uint16_t* gamma, float eps, int M, int N, int K, float* y, void* ws,
                    size_t ws_bytes, cudaStream_t stream) {
  const bool fused = pro != kern::kProInt8;
  const NextHint next = t_next;  // every call consumes the hint, launched or not
  t_next = NextHint{nullptr, 0, 0, 0, 0};
  if (M < 0 || M > max_m_for(bits) || N < 0 || K < 0 || K % kGroup || (long)M * K > kMaxMK) return WOQ_ERR_SHAPE;
  if (M == 0 || N == 0) return WOQ_OK;  // nothing to compute
  if (!y) return WOQ_ERR_NULL;
  if (!aligned(y, 4)) return WOQ_ERR_ALIGN;
  if (K == 0) {  // no groups: every output is the empty sum
    return cuda_result(cudaMemsetAsync(y, 0, (size_t)M * N * sizeof(float), stream));
  }
  if (!wpacked || !ws) return WOQ_ERR_NULL;
  if (fused ? !x : (!q || !ascale)) return WOQ_ERR_NULL;
  if (pro == kern::kProRms && !gamma) return WOQ_ERR_NULL;
  if (pro == kern::kProRms && !(eps >= 0.0f && eps <= 3.4028234e38f)) return WOQ_ERR_SHAPE;
  if (!aligned(wpacked, 16) || !aligned(y, 4) || !aligned(ws, 16)) return WOQ_ERR_ALIGN;
  if (fused ? !aligned(x, 16) : (!aligned(q, 16) || !aligned(ascale, 4))) return WOQ_ERR_ALIGN;
  if (pro == kern::kProRms && !aligned(gamma, 16)) return WOQ_ERR_ALIGN;
  if (wpacked_bytes < packed_bytes(bits, N, K)) return WOQ_ERR_LAYOUT;
  const LaunchConfig cfg = choose_config(bits, M, N, K, fused, pro == kern::kProSwiglu);
  if (cfg.ctas <= 0) return WOQ_ERR_SHAPE;
  const WorkspaceLayout wl = workspace_layout(M, N, K, cfg.ctas);
  if (ws_bytes < workspace_need(pro, wl) || cfg.ctas > max_ctas_for_workspace()) return WOQ_ERR_WORKSPACE;
  GemvParams p;
  p.w = static_cast<const uint8_t*>(wpacked);
  p.x = x;
  p.gamma = gamma;
  p.eps = eps;
  p.q = q;
  p.ascale = ascale;
  p.y = y;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  p.status = reinterpret_cast<uint32_t*>(wsb);
  p.parts = reinterpret_cast<unsigned long long*>(wsb + wl.parts_offset);
  p.sync = reinterpret_cast<uint32_t*>(wsb + kSyncOffset);
  // the scratch rows (SwiGLU prologue only) are the last M K 2 bytes of the caller's workspace
  // (16-byte aligned; ws_bytes >= wl.total puts them at or after wl.h_offset)
  p.hbuf = pro == kern::kProSwiglu
               ? reinterpret_cast<uint16_t*>(wsb + ((ws_bytes - (size_t)M * (size_t)K * 2) & ~(size_t)15))
               : nullptr;
  p.N = N;
  p.K = K;
  p.T = (N + kTileRows - 1) / kTileRows;
  p.G = K / kGroup;
  const unsigned long long nb64 = (unsigned long long)p.T * (unsigned long long)p.G;
  if ((nb64 + 1) * (unsigned long long)(cfg.ctas + 1) >= (1ull << 32)) return WOQ_ERR_SHAPE;  // 32-bit partition math
  p.NB = (uint32_t)nb64;
  p.div_c = FastDiv::make((uint32_t)cfg.ctas);
  p.div_nb = FastDiv::make(p.NB);
  p.div_g = FastDiv::make((uint32_t)p.G);
  p.stages = cfg.stages;
  p.prefetch_stages = cfg.prefetch_stages;
  p.act_stride = act_stride(K, cfg.consumer);
  p.act_offset = act_offset(M, K, fused, cfg.consumer);
  p.red_offset = red_offset(M, K, fused, cfg.consumer);
  p.ring_offset = ring_offset(M, K, fused, cfg.consumer);
  p.launch_id = g_launch_counter.fetch_add(1, std::memory_order_relaxed) & 0x7fffffff;
  plan_next_prefetch(p, next, M, fused);
  p.wait_ns = wait_bound_ns();
  const int fk = g_fault_kind.load(std::memory_order_relaxed);
  p.fault = (fk == 1 || fk == 2) ? fk : 0;
  p.fault_cta = (uint32_t)g_fault_cta.load(std::memory_order_relaxed);
  const cudaError_t e = launch_gemv_any(bits, pro, cfg.consumer, M, p, cfg, stream);
  return cuda_result(e);
}

int woq_prefetch_next(const void* next_wpacked, size_t next_wpacked_bytes, int bits, int N, int K, int budget_kb) {
  if (!next_wpacked) {
    t_next = NextHint{nullptr, 0, 0, 0, 0};
    return WOQ_OK;
  }
  if ((bits != 4 && bits != 6) || N < 0 || K < 0 || K % kGroup || budget_kb < 0 || budget_kb > 65536) return WOQ_ERR_SHAPE;
  if (!aligned(next_wpacked, 16)) return WOQ_ERR_ALIGN;
  if (next_wpacked_bytes < packed_bytes(bits, N, K)) return WOQ_ERR_LAYOUT;
  t_next = NextHint{next_wpacked, bits, N, K, budget_kb};
  return WOQ_OK;
}

int woq_w4a8_gemv(const void* wpacked, size_t wpacked_bytes, const int8_t* q, const float* ascale, int M, int N,
                  int K, float* y, void* ws, size_t ws_bytes, woq_stream_t stream) {
  return run_gemv(4, kern::kProInt8, wpacked, wpacked_bytes, nullptr, q, ascale, nullptr, 0.0f, M, N, K, y, ws,
                  ws_bytes, (cudaStream_t)stream);
}

int woq_w6a8_gemv(const void* wpacked, size_t wpacked_bytes, const int8_t* q, const float* ascale, int M, int N,
                  int K, float* y, void* ws, size_t ws_bytes, woq_stream_t stream) {
  return run_gemv(6, kern::kProInt8, wpacked, wpacked_bytes, nullptr, q, ascale, nullptr, 0.0f, M, N, K, y, ws,
                  ws_bytes, (cudaStream_t)stream);
}

int woq_w4a8_linear_bf16(const void* wpacked, size_t wpacked_bytes, const void* x_bf16, int M, int N, int K, float* y,
                         void* ws, size_t ws_bytes, woq_stream_t stream) {
  return run_gemv(4, kern::kProBf16, wpacked, wpacked_bytes, x_bf16, nullptr, nullptr, nullptr, 0.0f, M, N, K, y, ws,
                  ws_bytes, (cudaStream_t)stream);
}

int woq_w6a8_linear_bf16(const void* wpacked, size_t wpacked_bytes, const void* x_bf16, int M, int N, int K, float* y,
                         void* ws, size_t ws_bytes, woq_stream_t stream) {
  return run_gemv(6, kern::kProBf16, wpacked, wpacked_bytes, x_bf16, nullptr, nullptr, nullptr, 0.0f, M, N, K, y, ws,
                  ws_bytes, (cudaStream_t)stream);
}

int woq_w4a8_linear_rmsnorm_bf16(const void* wpacked, size_t wpacked_bytes, const void* x_bf16, const void* gamma_bf16,
                                 float eps, int M, int N, int K, float* y, void* ws, size_t ws_bytes,
                                 woq_stream_t stream) {
  return run_gemv(4, kern::kProRms, wpacked, wpacked_bytes, x_bf16, nullptr, nullptr,
                  static_cast<const uint16_t*>(gamma_bf16), eps, M, N, K, y, ws, ws_bytes, (cudaStream_t)stream);
}

int woq_w6a8_linear_rmsnorm_bf16(const void* wpacked, size_t wpacked_bytes, const void* x_bf16, const void* gamma_bf16,
                                 float eps, int M, int N, int K, float* y, void* ws, size_t ws_bytes,
                                 woq_stream_t stream) {
  return run_gemv(6, kern::kProRms, wpacked, wpacked_bytes, x_bf16, nullptr, nullptr,
                  static_cast<const uint16_t*>(gamma_bf16), eps, M, N, K, y, ws, ws_bytes, (cudaStream_t)stream);
}

int woq_w4a8_linear_swiglu_f32(const void* wpacked, size_t wpacked_bytes, const float* gate_up, int M, int N, int K,
                               float* y, void* ws, size_t ws_bytes, woq_stream_t stream) {
  return run_gemv(4, kern::kProSwiglu, wpacked, wpacked_bytes, gate_up, nullptr, nullptr, nullptr, 0.0f, M, N, K, y,
                  ws, ws_bytes, (cudaStream_t)stream);
}

int woq_w6a8_linear_swiglu_f32(const void* wpacked, size_t wpacked_bytes, const float* gate_up, int M, int N, int K,
                               float* y, void* ws, size_t ws_bytes, woq_stream_t stream) {
  return run_gemv(6, kern::kProSwiglu, wpacked, wpacked_bytes, gate_up, nullptr, nullptr, nullptr, 0.0f, M, N, K, y,
                  ws, ws_bytes, (cudaStream_t)stream);
}

int woq_debug_group_dots(int bits, const void* wpacked, size_t wpacked_bytes, const int8_t* q, int M, int N, int K,
                         int32_t* dots, woq_stream_t stream) {
  if ((bits != 4 && bits != 6) || M < 0 || M > kMaxM || N < 0 || K < 0 || K % kGroup) return WOQ_ERR_SHAPE;
  if (M == 0 || N == 0 || K == 0) return WOQ_OK;  // no groups or no outputs
  if (!wpacked || !q || !dots) return WOQ_ERR_NULL;
  if (!aligned(wpacked, 16) || !aligned(q, 16) || !aligned(dots, 4)) return WOQ_ERR_ALIGN;
  if (wpacked_bytes < packed_bytes(bits, N, K)) return WOQ_ERR_LAYOUT;
  return cuda_result(launch_group_dots(bits, wpacked, q, M, N, K, dots, (cudaStream_t)stream));
}

// ---------------------------------------------------------------------------
// Allocation-free variant of the int4 bf16 linear.
//
// Some callers cannot allocate device memory for a workspace: plugins that run inside
// a host application which owns every device allocation, and latency-critical loops
// with a fixed memory budget, where a cudaMalloc could synchronise the device or fail
// at run time.  This entry point needs no workspace from them: its scratch is a
// file-scope device array below, part of this library's image on every GPU that
// loads it and kept until the process exits.
static constexpr size_t kNoAllocScratchBytes = 2u << 20;  // 2 MiB
static constexpr size_t kNoAllocPartsOffset = 256;         // split-tile words: the workspace layout's parts_offset
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices];  // device address of g_noalloc_scratch, per device
}  // namespace

// Device address of the scratch array on the current device.  The array's name is only a
// host-side stand-in in host code, so the address is looked up once per device (with that
// device current) and cached.
static int noalloc_scratch(void** out) {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return WOQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[d] == nullptr) {
    void* ptr = nullptr;
    if (const cudaError_t e_ = cudaGetSymbolAddress(&ptr, g_noalloc_scratch); e_ != cudaSuccess) return cuda_result(e_);
    if (ptr == nullptr) return WOQ_ERR_CUDA;
    g_noalloc_ptr[d] = ptr;
  }
  *out = g_noalloc_ptr[d];
  return WOQ_OK;
}

#ifdef WOQ_TRACE
// Trace build only: the id the next GEMV / linear launch will get.
__attribute__((visibility("default"))) int woq_trace_next_launch_id(void) {
  return g_launch_counter.load() & 0x7fffffff;
}
#endif

int woq_w4a8_linear_bf16_noalloc(const void* wpacked, size_t wpacked_bytes, const void* x_bf16, int M, int N, int K,
                                 float* y, woq_stream_t stream) {
  if (M < 0 || M > kMaxM || N < 0 || K < 0 || K % kGroup || (long)M * K > kMaxMK) return WOQ_ERR_SHAPE;
  if (M == 0 || N == 0) return WOQ_OK;
  if (!y || (K > 0 && (!wpacked || !x_bf16))) return WOQ_ERR_NULL;
  if (!aligned(y, 4) || (K > 0 && (!aligned(wpacked, 16) || !aligned(x_bf16, 16)))) return WOQ_ERR_ALIGN;
  if (K > 0 && wpacked_bytes < packed_bytes(4, N, K)) return WOQ_ERR_LAYOUT;
  // the scratch this launch will use must fit in the static array (the same rule run_gemv applies)
  size_t need = 256;
  if (K > 0) {
    const LaunchConfig cfg = choose_config(4, M, N, K, true);
    if (cfg.ctas <= 0) return WOQ_ERR_SHAPE;
    if (cfg.ctas > max_ctas_for_workspace()) return WOQ_ERR_WORKSPACE;
    need = workspace_need(kern::kProBf16, workspace_layout(M, N, K, cfg.ctas));
  }
  if (need > kNoAllocScratchBytes) return WOQ_ERR_WORKSPACE;
  void* ws = nullptr;
  const int st = noalloc_scratch(&ws);
  if (st != WOQ_OK) return st;
  // The array keeps the previous call's contents: the split-tile words start from zero (no
  // allocation involved).  The status word (bytes 0 .. 3) is left alone: it keeps device-side
  // errors until woq_noalloc_read_status clears it.
  if (need > kNoAllocPartsOffset) {
    if (const cudaError_t e_ = cudaMemsetAsync(static_cast<uint8_t*>(ws) + kNoAllocPartsOffset, 0,
                                               need - kNoAllocPartsOffset, (cudaStream_t)stream);
        e_ != cudaSuccess)
      return cuda_result(e_);
  }
  return run_gemv(4, kern::kProBf16, wpacked, wpacked_bytes, x_bf16, nullptr, nullptr, nullptr, 0.0f, M, N, K, y, ws,
                  kNoAllocScratchBytes, (cudaStream_t)stream);
}

int woq_noalloc_read_status(int clear, uint32_t* status_out, woq_stream_t stream) {
  if (!status_out) return WOQ_ERR_NULL;
  void* ws = nullptr;
  const int st = noalloc_scratch(&ws);
  if (st != WOQ_OK) return st;
  return woq_read_status(ws, kNoAllocScratchBytes, clear, status_out, stream);
}

}  // extern "C"
