// The skinny GEMV / linear kernel for sm_103a.
//
// "Doubling LLM token rates in ComfyUI" (blog.comfy.org):
//   - "What is the bottleneck?": batch-of-one decode reads every weight once
//     per step with about one operation per weight, so the op is bound by the
//     weight-read bandwidth of the memory;
//   - "Optimizing the Linear Kernel": quantise the activation to int8, then a
//     GEMV over weights whose group scales are interleaved with them in the
//     order the kernel consumes them (each thread block streams one contiguous
//     run); dp4a (CUDA-core int8 dot products) for the inner product;
//   - "Paying attention to the attention!": the last block to finish combines
//     the partial results inside the same launch (used here for split tiles).
//
// GB300 design:
//   * One CTA per SM (persistent).  The matrix's blocks (128 rows x 128 k) are
//     dealt out as equal contiguous ranges, one per CTA, so every SM streams
//     the same number of bytes whatever N and K are.  A 128-row tile cut by a
//     range boundary is finished by the last of its CTAs to arrive (partial sums
//     in the workspace plus a ticket counter; no spin-waits, fixed summation
//     order, so results are deterministic).
//   * Warp 4 is the producer: one lane issues 1-D bulk copies (TMA engine) of
//     whole stages (4 consecutive blocks of one tile, 33 KB for int4) into a
//     ring of shared-memory stages, tracked by mbarriers, with an L2
//     evict-first policy since every weight byte is read once.
//   * Warps 0..3 consume: warp w takes block w of each stage.  Lane l owns rows
//     l, 32+l, 64+l, 96+l of the tile; for each 32-k quarter it reads its
//     16-byte chunk per row (consecutive lanes, conflict-free) and the quarter's
//     activations (same address for all lanes: a broadcast), unpacks int4 (or
//     int6) to int8 lanes with two masks and a shift, and runs dp4a.  Per group
//     the int32 dot is exact; the term (d * wscale) * ascale is formed with two
//     fp32 roundings, as in the definition, and accumulated in fp32.
//   * The activations (int8, M x K) sit in shared memory for the whole launch.
//     The fused entry quantises bf16 x itself (amax pass + quantise pass over x,
//     which is L2-resident), bit-identical to the standalone kernel.
//   * Programmatic dependent launch: the producer starts streaming weights
//     before the previous kernel in the stream has finished; consumers wait for
//     it (griddepcontrol.wait) before reading activations or writing anything.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "woq_device.cuh"
#include "woq_layout.h"

namespace woq {

struct GemvParams {
  const uint8_t* w;         // packed buffer (header first)
  const uint16_t* x;        // bf16 bits [M][K] (fused entry)
  const int8_t* q;          // int8 [M][K] (int8 entry)
  const float* ascale;      // fp32 [M] (int8 entry)
  float* y;                 // fp32 [M][N]
  uint32_t* status;         // workspace status word
  uint32_t* tickets;        // one counter per tile
  float* partials;          // [ctas][2][M][128]
  int N, K, T, G;
  long long NB;             // T * G blocks
  int stages;
  int act_offset;           // shared-memory offsets (bytes)
  int red_offset;
  int ring_offset;
};

namespace kern {

constexpr int kCW = 4;                 // consumer warps
constexpr int kConsumers = kCW * 32;   // 128 = rows per tile
constexpr int kSB = kCW;               // blocks per stage
constexpr int kBarConsumers = 1;       // named barrier id for the consumer warps

template <int BITS>
struct Fmt {
  static constexpr int kBlockBytes = BITS == 4 ? kBlockBytesW4 : kBlockBytesW6;
  static constexpr float kDotScale = BITS == 4 ? 0.0625f : 0.25f;  // lanes hold 16w (int4) or 4w (int6)
};

// first block of CTA c under an even split of NB blocks over C CTAs
__device__ __forceinline__ long long range_begin(long long c, long long NB, long long C) { return c * NB / C; }
// CTA whose range holds block b
__device__ __forceinline__ long long cta_of_block(long long b, long long NB, long long C) {
  return ((b + 1) * C - 1) / NB;
}

// int4 / int6 lanes of word i of a 16-byte chunk: lo covers k0..k0+3, hi k0+4..k0+7
template <int BITS>
__device__ __forceinline__ void unpack_word(uint32_t v, uint32_t uh, int e, uint32_t& lo, uint32_t& hi) {
  if constexpr (BITS == 4) {
    lo = (v << 4) & 0xF0F0F0F0u;
    hi = v & 0xF0F0F0F0u;
  } else {
    lo = ((v << 2) & 0x3C3C3C3Cu) | ((uh << (6 - 4 * e)) & 0xC0C0C0C0u);
    hi = ((v >> 2) & 0x3C3C3C3Cu) | ((uh << (4 - 4 * e)) & 0xC0C0C0C0u);
  }
}

// One block (128 rows x one group) by one warp: acc[j][m] += term(row 32j+lane, m).
template <int BITS, int M>
__device__ __forceinline__ void consume_block(const uint8_t* __restrict__ blk, const int8_t* __restrict__ act, int K,
                                              int g, int lane, const float (&as)[M], float (&acc)[4][M]) {
  const uint2 sc = *reinterpret_cast<const uint2*>(blk + 8 * lane);
  float wsc[4];
  wsc[0] = dev::half_bits_to_float(sc.x & 0xFFFFu) * Fmt<BITS>::kDotScale;
  wsc[1] = dev::half_bits_to_float(sc.x >> 16) * Fmt<BITS>::kDotScale;
  wsc[2] = dev::half_bits_to_float(sc.y & 0xFFFFu) * Fmt<BITS>::kDotScale;
  wsc[3] = dev::half_bits_to_float(sc.y >> 16) * Fmt<BITS>::kDotScale;

  int dot[4][M];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int m = 0; m < M; ++m) dot[j][m] = 0;

  const int8_t* ag = act + g * kGroup;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t a[M][8];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const uint4 a0 = *reinterpret_cast<const uint4*>(ag + (size_t)m * K + 32 * c);
      const uint4 a1 = *reinterpret_cast<const uint4*>(ag + (size_t)m * K + 32 * c + 16);
      a[m][0] = a0.x; a[m][1] = a0.y; a[m][2] = a0.z; a[m][3] = a0.w;
      a[m][4] = a1.x; a[m][5] = a1.y; a[m][6] = a1.z; a[m][7] = a1.w;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 v = *reinterpret_cast<const uint4*>(blk + kScaleBytes + ((c * 4 + j) * 32 + lane) * 16);
      uint2 u = make_uint2(0u, 0u);
      if constexpr (BITS == 6)
        u = *reinterpret_cast<const uint2*>(blk + kScaleBytes + kW4Bytes + ((c * 4 + j) * 32 + lane) * 8);
      const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t lo, hi;
        unpack_word<BITS>(vw[i], (i < 2) ? u.x : u.y, i & 1, lo, hi);
#pragma unroll
        for (int m = 0; m < M; ++m) {
          dot[j][m] = dev::dp4a_ss(lo, a[m][2 * i], dot[j][m]);
          dot[j][m] = dev::dp4a_ss(hi, a[m][2 * i + 1], dot[j][m]);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int m = 0; m < M; ++m) {
      // (d * wscale) * ascale with two fp32 roundings; lanes carry 16d (int4) or 4d (int6),
      // and wsc carries wscale / 16 (or / 4), so the first product is exactly fl(d * wscale)
      const float t = __fmul_rn(__fmul_rn(dev::small_int_to_float(dot[j][m]), wsc[j]), as[m]);
      acc[j][m] = __fadd_rn(acc[j][m], t);
    }
}

template <int BITS, int M, bool FUSED>
__global__ void __launch_bounds__(kConsumers + 32, 1) gemv_kernel(const GemvParams p) {
  constexpr int BB = Fmt<BITS>::kBlockBytes;
  constexpr int kStageBytes = kSB * BB;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + 8;
  float* s_as = reinterpret_cast<float*>(smem + 128);
  volatile int* s_flags = reinterpret_cast<volatile int*>(smem + 160);  // [0] ticket-last, [1] abort, [2] header-ok
  float* s_scratch = reinterpret_cast<float*>(smem + 192);               // [4 warps] amax partials
  int8_t* act = reinterpret_cast<int8_t*>(smem + p.act_offset);
  float* red = reinterpret_cast<float*>(smem + p.red_offset);
  uint8_t* ring = smem + p.ring_offset;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const long long C = gridDim.x;
  const long long cta = blockIdx.x;
  const long long b_begin = range_begin(cta, p.NB, C);
  const long long b_end = range_begin(cta + 1, p.NB, C);
  const int G = p.G;
  const int stages = p.stages;

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      dev::mbar_init(full + s, 1);
      dev::mbar_init(empty + s, kCW);
    }
    s_flags[0] = 0;
    s_flags[1] = 0;
    s_flags[2] = 1;
    dev::fence_mbar_init();
  }
  __syncthreads();
  // every CTA of this grid is resident (one per SM), so the next grid may be scheduled now
  dev::pdl_launch_dependents();

  if (warp == kCW) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = dev::l2_evict_first_policy();
      const uint8_t* blocks = p.w + kHeaderBytes;
      long long it = 0;
      bool ok = true;
      for (long long b = b_begin; b < b_end && ok;) {
        const long long t = b / G;
        const int g0 = (int)(b - t * G);
        const int gend = (int)((b_end < (t + 1) * G ? b_end : (t + 1) * G) - t * G);
        const int nb = gend - g0 < kSB ? gend - g0 : kSB;
        const int slot = (int)(it % stages);
        if (it >= stages && !dev::mbar_wait_bounded(empty + slot, (uint32_t)((it / stages - 1) & 1))) {
          ok = false;
          break;
        }
        const uint32_t bytes = (uint32_t)(nb * BB);
        dev::mbar_arrive_expect_tx(full + slot, bytes);
        dev::bulk_copy_g2s(ring + (size_t)slot * kStageBytes, blocks + (size_t)b * BB, bytes, full + slot, pol);
        ++it;
        b += nb;
      }
      if (!ok) atomicOr(p.status, 0x2u /* WOQ_DEVERR_TIMEOUT */);
      // no bulk copy may still be landing in this CTA's shared memory when it exits
      const long long first = it > stages ? it - stages : 0;
      for (long long i = first; i < it; ++i) dev::mbar_wait_bounded(full + (int)(i % stages), (uint32_t)((i / stages) & 1));
    }
    return;
  }

  // -------------------------------------------------------------------- consumers
  dev::pdl_wait_prior_grids();

  if (tid == 0) {
    // the packed header must describe this call's (bits, N, K)
    const uint4 h0 = *reinterpret_cast<const uint4*>(p.w);
    const uint4 h1 = *reinterpret_cast<const uint4*>(p.w + 16);
    const bool hok = h0.x == kMagic && h0.y == kLayoutVersion && h0.z == (uint32_t)BITS && h0.w == (uint32_t)kTileRows &&
                     h1.x == (uint32_t)p.N && h1.y == (uint32_t)p.K;
    if (!hok) {
      s_flags[2] = 0;
      atomicOr(p.status, 0x1u /* WOQ_DEVERR_HEADER */);
    }
  }

  // activations -> shared memory (int8, [M][K])
  if constexpr (FUSED) {
    // pass 1: amax per row; pass 2: q = rne(x / (amax / 127)), as the standalone kernel
#pragma unroll 1
    for (int m = 0; m < M; ++m) {
      const uint16_t* xr = p.x + (size_t)m * p.K;
      float amax = 0.0f;
      for (int e = tid * 8; e < p.K; e += kConsumers * 8) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr + e));
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          amax = fmaxf(amax, fabsf(dev::bf16_bits_to_float(w4[i] & 0xFFFFu)));
          amax = fmaxf(amax, fabsf(dev::bf16_bits_to_float(w4[i] >> 16)));
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (lane == 0) s_scratch[warp] = amax;
      dev::named_barrier_sync(kBarConsumers, kConsumers);
      amax = fmaxf(fmaxf(s_scratch[0], s_scratch[1]), fmaxf(s_scratch[2], s_scratch[3]));
      const float s = __fdiv_rn(amax, 127.0f);
      dev::named_barrier_sync(kBarConsumers, kConsumers);  // s_scratch is reused by the next row
      if (tid == 0) s_as[m] = s;
      for (int e = tid * 8; e < p.K; e += kConsumers * 8) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr + e));
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        uint32_t packed[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t bits16 = (i & 1) ? (w4[i >> 1] >> 16) : (w4[i >> 1] & 0xFFFFu);
          int qi = 0;
          if (s != 0.0f) {
            const float r = rintf(__fdiv_rn(dev::bf16_bits_to_float(bits16), s));
            qi = (int)fminf(fmaxf(r, -127.0f), 127.0f);
          }
          packed[i >> 2] |= ((uint32_t)qi & 0xFFu) << (8 * (i & 3));
        }
        *reinterpret_cast<uint2*>(act + (size_t)m * p.K + e) = make_uint2(packed[0], packed[1]);
      }
    }
  } else {
    const int mk16 = (M * p.K) >> 4;
    for (int i = tid; i < mk16; i += kConsumers)
      reinterpret_cast<uint4*>(act)[i] = __ldg(reinterpret_cast<const uint4*>(p.q) + i);
    if (tid < M) s_as[tid] = p.ascale[tid];
  }
  dev::named_barrier_sync(kBarConsumers, kConsumers);

  float as[M];
#pragma unroll
  for (int m = 0; m < M; ++m) as[m] = s_as[m];
  const bool header_ok = s_flags[2] != 0;

  const long long first_tile = b_begin / G;
  long long it = 0;
  int buf = 0;
  bool aborted = false;
  for (long long b = b_begin; b < b_end;) {
    const long long t = b / G;
    const int ga = (int)(b - t * G);
    const long long item_end = b_end < (t + 1) * G ? b_end : (t + 1) * G;
    const int gb = (int)(item_end - t * G);

    float acc[4][M];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int m = 0; m < M; ++m) acc[j][m] = 0.0f;

    for (int g0 = ga; g0 < gb; g0 += kSB) {
      const int nb = gb - g0 < kSB ? gb - g0 : kSB;
      const int slot = (int)(it % stages);
      if (!aborted && !dev::mbar_wait_bounded(full + slot, (uint32_t)((it / stages) & 1))) {
        aborted = true;
        s_flags[1] = 1;
        atomicOr(p.status, 0x2u /* WOQ_DEVERR_TIMEOUT */);
      }
      if (!aborted && warp < nb)
        consume_block<BITS, M>(ring + (size_t)slot * kStageBytes + (size_t)warp * BB, act, p.K, g0 + warp, lane, as,
                               acc);
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(empty + slot);
      ++it;
    }

    // reduce the four warps' partial sums for this tile: red[buf][warp][m][row]
    float* rb = red + (size_t)buf * (kCW * M * kTileRows);
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int m = 0; m < M; ++m) rb[(warp * M + m) * kTileRows + 32 * j + lane] = acc[j][m];
    dev::named_barrier_sync(kBarConsumers, kConsumers);
    const bool write_ok = header_ok && s_flags[1] == 0;
    const int row = tid;
    const long long n = t * kTileRows + row;
    float sum[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float s = rb[(0 * M + m) * kTileRows + row];
#pragma unroll
      for (int w = 1; w < kCW; ++w) s = __fadd_rn(s, rb[(w * M + m) * kTileRows + row]);
      sum[m] = s;
    }
    if (ga == 0 && gb == G) {
      if (write_ok && n < p.N) {
#pragma unroll
        for (int m = 0; m < M; ++m) p.y[(size_t)m * p.N + n] = sum[m];
      }
    } else {
      // tile split across CTAs: publish this CTA's part; the last to arrive sums all parts in CTA order.
      // Every consumer thread takes both barriers whatever write_ok says (no divergent bar.sync).
      const int part = (t == first_tile) ? 0 : 1;
      float* mine = p.partials + ((size_t)(cta * 2 + part) * M) * kTileRows;
      if (write_ok) {
#pragma unroll
        for (int m = 0; m < M; ++m) mine[m * kTileRows + row] = sum[m];
      }
      __threadfence();
      dev::named_barrier_sync(kBarConsumers, kConsumers);
      if (tid == 0) {
        int last = 0;
        if (write_ok) {
          const long long c_first = cta_of_block(t * G, p.NB, C);
          const long long c_last = cta_of_block(t * G + G - 1, p.NB, C);
          const unsigned parts = (unsigned)(c_last - c_first + 1);
          const unsigned prev = atomicAdd(p.tickets + t, 1u);
          last = prev == parts - 1;
          if (last) p.tickets[t] = 0u;  // ready for the next launch
        }
        s_flags[0] = last;
      }
      dev::named_barrier_sync(kBarConsumers, kConsumers);
      if (s_flags[0]) {
        __threadfence();
        const long long c_first = cta_of_block(t * G, p.NB, C);
        const long long c_last = cta_of_block(t * G + G - 1, p.NB, C);
        float tot[M];
#pragma unroll
        for (int m = 0; m < M; ++m) tot[m] = 0.0f;
        for (long long c2 = c_first; c2 <= c_last; ++c2) {
          const int part2 = (t == range_begin(c2, p.NB, C) / G) ? 0 : 1;
          const float* src = p.partials + ((size_t)(c2 * 2 + part2) * M) * kTileRows;
#pragma unroll
          for (int m = 0; m < M; ++m) tot[m] = __fadd_rn(tot[m], __ldcg(src + m * kTileRows + row));
        }
        if (n < p.N) {
#pragma unroll
          for (int m = 0; m < M; ++m) p.y[(size_t)m * p.N + n] = tot[m];
        }
      }
    }
    buf ^= 1;
    b = item_end;
  }
}

}  // namespace kern
}  // namespace woq
