// Small kernels: standalone activation quantisation, the debug group-dot
// kernel and the device-side packer.
#include <cuda_fp16.h>

#include "woq_device.cuh"
#include "woq_gemv.cuh"
#include "woq_internal.h"
#include "woq_layout.h"

namespace woq {
namespace kern {

// ---------------------------------------------------------------------------
// Activation quantisation ("Optimizing the Linear Kernel": the activation is
// quantised to int8 before the linear).  One CTA per row:
// amax = max |x|; s = amax / 127 (IEEE); q = rne(x / s) (IEEE), clamped to
// [-127, 127]; a zero row gives s = 0 and q = 0.
// ---------------------------------------------------------------------------
constexpr int kAqThreads = 1024;

__device__ __forceinline__ int8_t quant_one(float x, float s) {
  if (s == 0.0f) return 0;
  const float r = rintf(__fdiv_rn(x, s));
  return (int8_t)(int)fminf(fmaxf(r, -127.0f), 127.0f);
}

__global__ void __launch_bounds__(kAqThreads) act_quant_kernel(const uint16_t* __restrict__ x, int K,
                                                               int8_t* __restrict__ q, float* __restrict__ ascale) {
  __shared__ float s_part[kAqThreads / 32];
  dev::pdl_launch_dependents();
  dev::pdl_wait_prior_grids();
  const int m = blockIdx.x;
  const int tid = threadIdx.x;
  const uint16_t* xr = x + (size_t)m * K;
  int8_t* qr = q + (size_t)m * K;
  const bool vec = (K % 8) == 0;
  float amax = 0.0f;
  if (vec) {
    for (int e = tid * 8; e < K; e += kAqThreads * 8) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr + e));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        amax = fmaxf(amax, fabsf(dev::bf16_bits_to_float(w[i] & 0xFFFFu)));
        amax = fmaxf(amax, fabsf(dev::bf16_bits_to_float(w[i] >> 16)));
      }
    }
  } else {
    for (int e = tid; e < K; e += kAqThreads) amax = fmaxf(amax, fabsf(dev::bf16_bits_to_float(xr[e])));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((tid & 31) == 0) s_part[tid >> 5] = amax;
  __syncthreads();
  amax = s_part[0];
  for (int i = 1; i < kAqThreads / 32; ++i) amax = fmaxf(amax, s_part[i]);
  const float s = __fdiv_rn(amax, 127.0f);
  if (tid == 0) ascale[m] = s;
  if (vec) {
    for (int e = tid * 8; e < K; e += kAqThreads * 8) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr + e));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t packed[2] = {0u, 0u};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t b16 = (i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xFFFFu);
        packed[i >> 2] |= ((uint32_t)(uint8_t)quant_one(dev::bf16_bits_to_float(b16), s)) << (8 * (i & 3));
      }
      *reinterpret_cast<uint2*>(qr + e) = make_uint2(packed[0], packed[1]);
    }
  } else {
    for (int e = tid; e < K; e += kAqThreads) qr[e] = quant_one(dev::bf16_bits_to_float(xr[e]), s);
  }
}

// ---------------------------------------------------------------------------
// Standalone RMSNorm / SwiGLU followed by activation quantisation (the unfused
// form of the linear's prologue fusions, same arithmetic: woq_prologue.cuh).
// One CTA per row; h is formed in shared memory (bf16 [K]) and quantised as by
// act_quant_kernel.  K % 8 == 0.
// ---------------------------------------------------------------------------
template <int PRO>
__global__ void __launch_bounds__(kAqThreads) pro_act_quant_kernel(const void* __restrict__ x,
                                                                   const uint16_t* __restrict__ gamma, float eps,
                                                                   int K, int8_t* __restrict__ q,
                                                                   float* __restrict__ ascale) {
  extern __shared__ __align__(16) uint16_t s_h[];  // [K]
  __shared__ float s_part[kAqThreads / 32];
  __shared__ uint32_t s_bits;
  __shared__ unsigned long long s_sum;
  dev::pdl_launch_dependents();
  dev::pdl_wait_prior_grids();
  const int m = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31;
  if (PRO == kProRms) {
    const uint16_t* xr = static_cast<const uint16_t*>(x) + (size_t)m * K;
    if (tid == 0) {
      s_bits = 0u;
      s_sum = 0ull;
    }
    __syncthreads();
    uint32_t acc = 0;
    for (int e = tid * 8; e < K; e += kAqThreads * 8) acc = absmax8(acc, __ldg(reinterpret_cast<const uint4*>(xr + e)));
    const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(dev::bf16x2_absmax_to_float(acc)));
    if (lane == 0) atomicMax(&s_bits, wm);
    __syncthreads();
    const int C = pro::rms_row_exponent(s_bits);
    unsigned long long part = 0;
    if (C != -1000) {
      for (int e = tid * 8; e < K; e += kAqThreads * 8) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr + e));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) part += pro::rms_term(w[i] & 0xFFFFu, C) + pro::rms_term(w[i] >> 16, C);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0 && part) atomicAdd(&s_sum, part);
    __syncthreads();
    const float r = C == -1000 ? 0.0f : pro::rms_rcp(s_sum, C, K, eps);
    for (int e = tid * 8; e < K; e += kAqThreads * 8)
      *reinterpret_cast<uint4*>(s_h + e) = pro::rms_h8(__ldg(reinterpret_cast<const uint4*>(xr + e)),
                                                       __ldg(reinterpret_cast<const uint4*>(gamma + e)), r);
  } else {
    const float* g = static_cast<const float*>(x) + (size_t)m * 2 * K;
    const float* u = g + K;
    for (int e = tid; e < K; e += kAqThreads) s_h[e] = (uint16_t)pro::swiglu_bf16(__ldg(g + e), __ldg(u + e));
  }
  __syncthreads();
  // quantise h as act_quant_kernel quantises x
  float amax = 0.0f;
  for (int e = tid; e < K; e += kAqThreads) amax = fmaxf(amax, fabsf(dev::bf16_bits_to_float(s_h[e])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) s_part[tid >> 5] = amax;
  __syncthreads();
  amax = s_part[0];
  for (int i = 1; i < kAqThreads / 32; ++i) amax = fmaxf(amax, s_part[i]);
  const float s = __fdiv_rn(amax, 127.0f);
  if (tid == 0) ascale[m] = s;
  int8_t* qr = q + (size_t)m * K;
  for (int e = tid; e < K; e += kAqThreads) qr[e] = quant_one(dev::bf16_bits_to_float(s_h[e]), s);
}

// ---------------------------------------------------------------------------
// Debug: exact per-group dot products straight from the packed layout.
// One thread per (row n, group g); dots[m][n][g].
// ---------------------------------------------------------------------------
template <int BITS, int M>
__global__ void group_dots_kernel(const uint8_t* __restrict__ w, const int8_t* __restrict__ q, int N, int K,
                                  int32_t* __restrict__ dots) {
  constexpr int BB = Fmt<BITS>::kBlockBytes;
  const int G = K / kGroup;
  const long long total = (long long)N * G;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int n = (int)(idx / G);
    const int g = (int)(idx % G);
    const int t = n / kTileRows, r = n % kTileRows, j = r / 32, l = r % 32;
    const uint8_t* blk = w + kHeaderBytes + ((size_t)t * G + g) * BB;
    int d[M];
#pragma unroll
    for (int m = 0; m < M; ++m) d[m] = 0;
    for (int c = 0; c < 4; ++c) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(blk + w4_chunk_offset(c, j, l)));
      uint2 u = make_uint2(0u, 0u);
      if constexpr (BITS == 6)
        u = __ldg(reinterpret_cast<const uint2*>(blk + hi_chunk_offset(c, j, l)));
      const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t lo, hi;
        unpack_word<BITS>(vw[i], (i < 2) ? u.x : u.y, i & 1, lo, hi);
        const int k0 = g * kGroup + 32 * c + 8 * i;
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const uint2 a = __ldg(reinterpret_cast<const uint2*>(q + (size_t)m * K + k0));
          d[m] = dev::dp4a_ss(lo, a.x, d[m]);
          d[m] = dev::dp4a_ss(hi, a.y, d[m]);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < M; ++m) dots[((size_t)m * N + n) * G + g] = BITS == 4 ? (d[m] >> 4) : (d[m] >> 2);
  }
}

// ---------------------------------------------------------------------------
// Device packer: one thread per (tile, group, quarter c, row group j, lane l)
// chunk; writes the same bytes as the host packer.
// ---------------------------------------------------------------------------
__host__ __device__ inline size_t canonical_row_bytes(int bits, int K) {
  return bits == 4 ? (size_t)K / 2 : (size_t)K / 4 * 3;
}

// The packed words of one chunk (one row, one 32-k quarter) from its canonical bytes:
// 16 bytes of int4 (two per byte, low nibble = even k) or 24 bytes of int6 (four per
// three bytes).  lo: the int4 / low-nibble words, hi: the int6 high-bit words.
// The canonical bytes of one chunk (32 weights of one row): 16 (int4) or 24 (int6) bytes.
struct RawChunk {
  uint32_t w[6];
};
template <int BITS>
__device__ __forceinline__ RawChunk load_chunk(const uint8_t* __restrict__ src) {
  RawChunk r = {{0u, 0u, 0u, 0u, 0u, 0u}};
  if constexpr (BITS == 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(src);
    r.w[0] = v.x, r.w[1] = v.y, r.w[2] = v.z, r.w[3] = v.w;
  } else {
    const uint2 a = *reinterpret_cast<const uint2*>(src);
    const uint2 b = *reinterpret_cast<const uint2*>(src + 8);
    const uint2 cc = *reinterpret_cast<const uint2*>(src + 16);
    r.w[0] = a.x, r.w[1] = a.y, r.w[2] = b.x, r.w[3] = b.y, r.w[4] = cc.x, r.w[5] = cc.y;
  }
  return r;
}

// A chunk's canonical bytes -> its packed words (lo: the int4 region's 16 bytes; hi: the
// int6 top-bit plane's 8 bytes).
template <int BITS>
__device__ __forceinline__ void convert_chunk(const RawChunk& raw, uint32_t (&lo)[4], uint32_t (&hi)[2]) {
  uint8_t code[32];
  if constexpr (BITS == 4) {
    const uint32_t* vw = raw.w;
#pragma unroll
    for (int kk = 0; kk < 32; ++kk) code[kk] = (uint8_t)((vw[kk >> 3] >> (4 * (kk & 7))) & 0xF);
  } else {
    const uint32_t* bw = raw.w;
#pragma unroll
    for (int quad = 0; quad < 8; ++quad) {
      uint32_t word = 0;
#pragma unroll
      for (int byte = 0; byte < 3; ++byte) {
        const int pos = quad * 3 + byte;
        word |= ((bw[pos >> 2] >> (8 * (pos & 3))) & 0xFFu) << (8 * byte);
      }
#pragma unroll
      for (int f = 0; f < 4; ++f) code[quad * 4 + f] = (uint8_t)((word >> (6 * f)) & 0x3F);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    lo[i] = 0u;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint8_t ca = code[8 * i + b], cb = code[8 * i + 4 + b];
      lo[i] |= ((uint32_t)(ca & 0xF) | ((uint32_t)(cb & 0xF) << 4)) << (8 * b);
    }
  }
  hi[0] = hi[1] = 0u;
  if constexpr (BITS == 6) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint8_t ca = code[8 * i + b], cb = code[8 * i + 4 + b];
        const int h = i >> 1, e = i & 1;
        hi[h] |= ((uint32_t)((ca >> 4) & 3) << (2 * (2 * e))) << (8 * b);
        hi[h] |= ((uint32_t)((cb >> 4) & 3) << (2 * (2 * e + 1))) << (8 * b);
      }
  }
}

template <int BITS>
__device__ __forceinline__ void pack_chunk(const uint8_t* __restrict__ src, uint32_t (&lo)[4], uint32_t (&hi)[2]) {
  convert_chunk<BITS>(load_chunk<BITS>(src), lo, hi);
}
template <int BITS>
__global__ void pack_kernel(const uint8_t* __restrict__ q, const uint16_t* __restrict__ scales, int N, int K, int T,
                            uint8_t* __restrict__ dst, PackedHeader hdr) {
  constexpr int BB = Fmt<BITS>::kBlockBytes;
  const int G = K / kGroup;
  const long long total = (long long)T * G * 512;
  if (blockIdx.x == 0 && threadIdx.x < kHeaderBytes / 4) {
    uint32_t word = 0;
    if (threadIdx.x * 4 < (int)sizeof(PackedHeader)) memcpy(&word, reinterpret_cast<const uint8_t*>(&hdr) + threadIdx.x * 4, 4);
    reinterpret_cast<uint32_t*>(dst)[threadIdx.x] = word;
  }
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int l = (int)(idx & 31);
    const int j = (int)((idx >> 5) & 3);
    const int c = (int)((idx >> 7) & 3);
    const long long tg = idx >> 9;
    const int g = (int)(tg % G);
    const long long t = tg / G;
    const long long n = t * kTileRows + 32 * j + l;
    uint8_t* blk = dst + kHeaderBytes + (size_t)tg * BB;
    uint32_t lo[4] = {0u, 0u, 0u, 0u};
    uint32_t hi[2] = {0u, 0u};
    if (n < N) {
      const int kb = g * kGroup + 32 * c;
      pack_chunk<BITS>(q + (size_t)n * canonical_row_bytes(BITS, K) + (size_t)kb * BITS / 8, lo, hi);
    }
    *reinterpret_cast<uint4*>(blk + w4_chunk_offset(c, j, l)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    if constexpr (BITS == 6)
      *reinterpret_cast<uint2*>(blk + hi_chunk_offset(c, j, l)) = make_uint2(hi[0], hi[1]);
    if (c == 0) {
      const int r = 32 * j + l;
      const uint16_t s = n < N ? scales[(size_t)n * G + g] : (uint16_t)0;
      reinterpret_cast<uint16_t*>(blk)[scale_index(r)] = s;
    }
  }
}

// ---------------------------------------------------------------------------
// In-place relayout ("Optimizing the Linear Kernel": the weights are rearranged inside
// the device buffer that holds them, once when the model is loaded, without a second
// buffer on the device or the host).  The buffer holds, from byte
// 256 on, the canonical weights (N rows) directly followed by the canonical fp16 scales;
// it ends up holding the packed layout.  A packed tile t starts at 256 + t G BB, never
// below the canonical bytes of any lower tile (G BB >= 128 row bytes), so the tiles are
// rewritten in batches of whole tiles from the top down: every CTA first copies all the
// scales it will write into shared memory (the top tiles overwrite the scale region),
// then per batch gathers its blocks' canonical chunks (a contiguous run of the batch's
// blocks, so rows are read in long segments), converted to the packed order,
// into shared memory, meets the other CTAs at a grid barrier (every read of the batch is
// done) and writes them out.  The 256-byte header slot holds the barrier words (0: arrivals,
// 1: generation, 2: failure, 3: departures) until CTA 0, once every CTA has counted its
// last write, writes the header over them.  One CTA per SM, launched cooperatively (all
// resident); every wait is bounded, and a wait that runs out sets word 2 and ends its CTA,
// so the header is never written.
// ---------------------------------------------------------------------------
constexpr int kRlThreads = 512;  // one thread per chunk of a block

struct RelayoutPlan {
  int N, K, T, G;
  int tiles_per_batch;  // whole tiles per batch, batches from the top down
  int q_slots;          // blocks a CTA stages per batch
  int scale_slots;      // blocks whose scales a CTA stages for the whole run
  unsigned long long wait_ns;  // bound of every wait on the other CTAs
  int fault_cta;               // tests of that bound: this CTA leaves before the first barrier (-1: none)
};


// Grid barrier on words[0] (arrivals) and words[1] (generation); bounded.
__device__ bool rl_grid_barrier(uint32_t* words, int* s_ok, unsigned long long wait_ns) {
  __syncthreads();
  if (threadIdx.x == 0) {
    bool ok = true;
    const uint32_t gen = dev::ld_acquire_u32(words + 1);
    __threadfence();
    if (atomicAdd(words, 1u) == gridDim.x - 1) {
      atomicExch(words, 0u);
      __threadfence();
      dev::st_release_u32(words + 1, gen + 1);
    } else {
      const uint64_t t0 = dev::global_timer_ns();
      while (dev::ld_acquire_u32(words + 1) == gen) {
        if (dev::global_timer_ns() - t0 > wait_ns) {
          ok = false;
          break;
        }
        __nanosleep(128);
      }
    }
    if (!ok) atomicExch(words + 2, 1u);
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

template <int BITS>
__global__ void __launch_bounds__(kRlThreads) relayout_kernel(uint8_t* buf, RelayoutPlan pl, PackedHeader hdr) {
  constexpr int BB = Fmt<BITS>::kBlockBytes;
  constexpr int QB = BB - kScaleBytes;  // weight bytes of a block
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* s_scales = reinterpret_cast<uint16_t*>(smem);              // [scale_slots][128], packed order
  uint8_t* s_q = smem + (size_t)pl.scale_slots * kScaleBytes;          // [q_slots][QB], packed order
  __shared__ int s_ok;
  uint32_t* words = reinterpret_cast<uint32_t*>(buf);
  const uint8_t* canon_q = buf + kHeaderBytes;
  const size_t R = canonical_row_bytes(BITS, pl.K);
  const uint16_t* canon_s = reinterpret_cast<const uint16_t*>(canon_q + (size_t)pl.N * R);
  const int C = (int)gridDim.x, cta = (int)blockIdx.x, tid = (int)threadIdx.x;

  // every scale this CTA will write, in the order it will write them
  int slot = 0;
  for (int thi = pl.T; thi > 0; thi -= pl.tiles_per_batch) {
    const int tlo = thi > pl.tiles_per_batch ? thi - pl.tiles_per_batch : 0;
    const int nb = (thi - tlo) * pl.G;
    const int i_lo = (int)((long long)cta * nb / C), i_hi = (int)((long long)(cta + 1) * nb / C);
    // thread (block offset tid / 128, row tid % 128): four blocks per pass, kSU passes' loads
    // in flight before their stores
    constexpr int kBPP = kRlThreads / kTileRows, kSU = 8;
    const int r = tid % kTileRows;
    for (int i0 = i_lo; i0 < i_hi; i0 += kBPP * kSU) {
      uint16_t v[kSU];
#pragma unroll
      for (int u = 0; u < kSU; ++u) {
        const int i = i0 + u * kBPP + tid / kTileRows;
        v[u] = 0;
        if (i < i_hi) {
          const int b = tlo * pl.G + i, t = b / pl.G, g = b % pl.G;
          const int n = t * kTileRows + r;
          if (n < pl.N) v[u] = canon_s[(size_t)n * pl.G + g];
        }
      }
#pragma unroll
      for (int u = 0; u < kSU; ++u) {
        const int i = i0 + u * kBPP + tid / kTileRows;
        if (i < i_hi) s_scales[(slot + (i - i_lo)) * kTileRows + scale_index(r)] = v[u];
      }
    }
    slot += i_hi - i_lo;
  }
  if (cta == pl.fault_cta) return;  // injected fault: never arrives, the others' waits run out
  if (!rl_grid_barrier(words, &s_ok, pl.wait_ns)) return;

  slot = 0;
  // this thread's chunk of every block: four consecutive lanes take the four 32-k quarters of
  // one row, so a warp reads eight rows' contiguous 64 (int4) or 96 (int6) bytes of the group
  const int c4 = tid & 3, r = tid >> 2, j = r >> 5, l = r & 31;
  for (int thi = pl.T; thi > 0; thi -= pl.tiles_per_batch) {
    const int tlo = thi > pl.tiles_per_batch ? thi - pl.tiles_per_batch : 0;
    const int nb = (thi - tlo) * pl.G;
    const int i_lo = (int)((long long)cta * nb / C), i_hi = (int)((long long)(cta + 1) * nb / C);
    // gather, converted to the packed order; kUnroll blocks' loads in flight before converting
    constexpr int kUnroll = 8;
    for (int i0 = i_lo, k0 = 0; i0 < i_hi; i0 += kUnroll, k0 += kUnroll) {
      RawChunk raw[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int i = i0 + u;
        raw[u] = RawChunk{{0u, 0u, 0u, 0u, 0u, 0u}};
        if (i < i_hi) {
          const int b = tlo * pl.G + i, t = b / pl.G, g = b % pl.G;
          const int n = t * kTileRows + 32 * j + l;
          if (n < pl.N) raw[u] = load_chunk<BITS>(canon_q + (size_t)n * R + (size_t)(g * kGroup + 32 * c4) * BITS / 8);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (i0 + u >= i_hi) break;
        uint32_t lo[4], hi[2];
        convert_chunk<BITS>(raw[u], lo, hi);
        uint8_t* sb = s_q + (size_t)(k0 + u) * QB - kScaleBytes;  // chunk offsets count from the block start
        *reinterpret_cast<uint4*>(sb + w4_chunk_offset(c4, j, l)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        if constexpr (BITS == 6)
          *reinterpret_cast<uint2*>(sb + hi_chunk_offset(c4, j, l)) = make_uint2(hi[0], hi[1]);
      }
    }
    if (!rl_grid_barrier(words, &s_ok, pl.wait_ns)) return;  // every canonical byte of the batch has been read
    int k = 0;
    for (int i = i_lo; i < i_hi; ++i, ++k, ++slot) {
      uint8_t* out = buf + kHeaderBytes + (size_t)(tlo * pl.G + i) * BB;
      for (int e = tid; e < kScaleBytes / 16; e += kRlThreads)
        reinterpret_cast<uint4*>(out)[e] = reinterpret_cast<const uint4*>(s_scales + (size_t)slot * kTileRows)[e];
      for (int e = tid; e < QB / 16; e += kRlThreads)
        reinterpret_cast<uint4*>(out + kScaleBytes)[e] = reinterpret_cast<const uint4*>(s_q + (size_t)k * QB)[e];
    }
  }
  __syncthreads();
  if (tid == 0) {  // count this CTA's writes as done
    __threadfence();
    atomicAdd(words + 3, 1u);
  }
  if (cta != 0) return;
  if (tid == 0) {  // CTA 0 waits for every CTA, so nobody still reads the barrier words
    bool ok = true;
    const uint64_t t0 = dev::global_timer_ns();
    while (dev::ld_acquire_u32(words + 3) != (uint32_t)C) {
      if (dev::global_timer_ns() - t0 > pl.wait_ns) {
        ok = false;
        break;
      }
      __nanosleep(128);
    }
    if (!ok) atomicExch(words + 2, 1u);
    s_ok = ok;
  }
  __syncthreads();
  if (!s_ok) return;
  if (tid < kHeaderBytes / 4) {  // the header last, over the barrier words
    uint32_t word = 0;
    if (tid * 4 < (int)sizeof(PackedHeader)) memcpy(&word, reinterpret_cast<const uint8_t*>(&hdr) + tid * 4, 4);
    words[tid] = word;
  }
}

}  // namespace kern

static cudaError_t launch_pdl(const void* func, dim3 grid, dim3 block, cudaStream_t stream, void** args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = 0;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelExC(&lc, func, args);
}

cudaError_t launch_act_quant(const void* x_bf16, int M, int K, int8_t* q, float* ascale, cudaStream_t stream) {
  const uint16_t* x = static_cast<const uint16_t*>(x_bf16);
  void* args[] = {(void*)&x, (void*)&K, (void*)&q, (void*)&ascale};
  return launch_pdl((const void*)kern::act_quant_kernel, dim3((unsigned)M), dim3(kern::kAqThreads), stream, args);
}

cudaError_t launch_pro_act_quant(int pro, const void* x, const uint16_t* gamma, float eps, int M, int K, int8_t* q,
                                 float* ascale, cudaStream_t stream) {
  const void* func = pro == kern::kProRms ? (const void*)kern::pro_act_quant_kernel<kern::kProRms>
                                          : (const void*)kern::pro_act_quant_kernel<kern::kProSwiglu>;
  const size_t smem = (size_t)K * 2;
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  void* args[] = {(void*)&x, (void*)&gamma, (void*)&eps, (void*)&K, (void*)&q, (void*)&ascale};
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)M);
  lc.blockDim = dim3(kern::kAqThreads);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelExC(&lc, func, args);
}

template <int BITS>
static cudaError_t launch_dots_bits(const void* wpacked, const int8_t* q, int M, int N, int K, int32_t* dots,
                                    cudaStream_t stream) {
  const uint8_t* w = static_cast<const uint8_t*>(wpacked);
  const long long total = (long long)N * (K / kGroup);
  const int threads = 256;
  const long long blocks_needed = (total + threads - 1) / threads;
  const unsigned blocks = (unsigned)(blocks_needed < 65535 ? blocks_needed : 65535);
  switch (M) {
    case 1: kern::group_dots_kernel<BITS, 1><<<blocks, threads, 0, stream>>>(w, q, N, K, dots); break;
    case 2: kern::group_dots_kernel<BITS, 2><<<blocks, threads, 0, stream>>>(w, q, N, K, dots); break;
    case 3: kern::group_dots_kernel<BITS, 3><<<blocks, threads, 0, stream>>>(w, q, N, K, dots); break;
    case 4: kern::group_dots_kernel<BITS, 4><<<blocks, threads, 0, stream>>>(w, q, N, K, dots); break;
    case 5: kern::group_dots_kernel<BITS, 5><<<blocks, threads, 0, stream>>>(w, q, N, K, dots); break;
    case 6: kern::group_dots_kernel<BITS, 6><<<blocks, threads, 0, stream>>>(w, q, N, K, dots); break;
    case 7: kern::group_dots_kernel<BITS, 7><<<blocks, threads, 0, stream>>>(w, q, N, K, dots); break;
    case 8: kern::group_dots_kernel<BITS, 8><<<blocks, threads, 0, stream>>>(w, q, N, K, dots); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_group_dots(int bits, const void* wpacked, const int8_t* q, int M, int N, int K, int32_t* dots,
                              cudaStream_t stream) {
  return bits == 4 ? launch_dots_bits<4>(wpacked, q, M, N, K, dots, stream)
                   : launch_dots_bits<6>(wpacked, q, M, N, K, dots, stream);
}

cudaError_t launch_pack_device(int bits, const uint8_t* q, const uint16_t* scales, int N, int K, void* dst,
                               cudaStream_t stream) {
  const int T = (N + kTileRows - 1) / kTileRows;
  const int G = K / kGroup;
  PackedHeader h;
  memset(&h, 0, sizeof(h));
  h.magic = kMagic;
  h.version = kLayoutVersion;
  h.bits = (uint32_t)bits;
  h.tile_rows = kTileRows;
  h.N = (uint32_t)N;
  h.K = (uint32_t)K;
  h.tiles = (uint32_t)T;
  h.groups = (uint32_t)G;
  h.block_bytes = (uint64_t)block_bytes(bits);
  h.total_bytes = (uint64_t)packed_bytes(bits, N, K);
  const long long total = (long long)T * G * 512;
  const int threads = 256;
  long long blocks_needed = (total + threads - 1) / threads;
  if (blocks_needed < 1) blocks_needed = 1;
  const unsigned blocks = (unsigned)(blocks_needed < 1048576 ? blocks_needed : 1048576);
  uint8_t* d = static_cast<uint8_t*>(dst);
  if (bits == 4)
    kern::pack_kernel<4><<<blocks, threads, 0, stream>>>(q, scales, N, K, T, d, h);
  else
    kern::pack_kernel<6><<<blocks, threads, 0, stream>>>(q, scales, N, K, T, d, h);
  return cudaGetLastError();
}

}  // namespace woq


namespace woq {

// Relayout plan: batches of whole tiles whose staged blocks fit next to all of the CTA's
// staged scales; 0 tiles per batch if even one tile does not fit.
static kern::RelayoutPlan relayout_plan(int bits, int N, int K, int ctas, int smem) {
  kern::RelayoutPlan pl = {N, K, (N + kTileRows - 1) / kTileRows, K / kGroup, 0, 0, 0, dev::kWaitLimitNs, -1};
  const int QB = block_bytes(bits) - kScaleBytes;
  for (int tb = pl.T; tb >= 1; --tb) {
    int scale_slots = 0, q_slots = 0;
    for (int thi = pl.T; thi > 0; thi -= tb) {
      const int tlo = thi > tb ? thi - tb : 0;
      const int per = ((thi - tlo) * pl.G + ctas - 1) / ctas;
      scale_slots += per;
      if (per > q_slots) q_slots = per;
    }
    if ((long long)scale_slots * kScaleBytes + (long long)q_slots * QB <= smem) {
      pl.tiles_per_batch = tb;
      pl.q_slots = q_slots;
      pl.scale_slots = scale_slots;
      return pl;
    }
  }
  return pl;
}

cudaError_t launch_relayout(int bits, void* buf, int N, int K, int* too_large, cudaStream_t stream,
                            unsigned long long wait_ns, int fault_cta) {
  *too_large = 0;
  int dev = 0, sms = 0, smem = 0, coop = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  if (e != cudaSuccess) return e;
  if (!coop) return cudaErrorNotSupported;
  const int budget = smem - 1024;  // static shared memory and slack
  const kern::RelayoutPlan pl = relayout_plan(bits, N, K, sms, budget);
  if (pl.tiles_per_batch <= 0) {
    *too_large = 1;
    return cudaSuccess;
  }
  PackedHeader h;
  memset(&h, 0, sizeof(h));
  h.magic = kMagic;
  h.version = kLayoutVersion;
  h.bits = (uint32_t)bits;
  h.tile_rows = kTileRows;
  h.N = (uint32_t)N;
  h.K = (uint32_t)K;
  h.tiles = (uint32_t)pl.T;
  h.groups = (uint32_t)pl.G;
  h.block_bytes = (uint64_t)block_bytes(bits);
  h.total_bytes = (uint64_t)packed_bytes(bits, N, K);
  const void* func = bits == 4 ? (const void*)kern::relayout_kernel<4> : (const void*)kern::relayout_kernel<6>;
  const size_t dyn = (size_t)pl.scale_slots * kScaleBytes + (size_t)pl.q_slots * (block_bytes(bits) - kScaleBytes);
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, func, kern::kRlThreads, dyn);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  // the barrier words live in the header slot: start them at zero
  e = cudaMemsetAsync(buf, 0, kHeaderBytes, stream);
  if (e != cudaSuccess) return e;
  uint8_t* b = static_cast<uint8_t*>(buf);
  kern::RelayoutPlan plan = pl;
  plan.wait_ns = wait_ns;
  plan.fault_cta = fault_cta;
  void* args[] = {(void*)&b, (void*)&plan, (void*)&h};
  return cudaLaunchCooperativeKernel(func, dim3((unsigned)sms), dim3(kern::kRlThreads), args, dyn, stream);
}

}  // namespace woq
