// The skinny GEMV / linear kernel for sm_103a.
//
// "Doubling LLM token rates in ComfyUI" (blog.comfy.org):
//   - "What is the bottleneck?": batch-of-one decode reads every weight once
//     per step with about one operation per weight, so the op is bound by the
//     weight-read bandwidth of the memory;
//   - "Optimizing the Linear Kernel": quantise the activation to int8, then a
//     GEMV reading weights and their group scales from one buffer arranged in
//     reading order (a contiguous run per thread block); dp4a (CUDA-core int8
//     dot products) for the inner product;
//   - "Paying attention to the attention!": partial results are merged inside
//     the launch that produced them (used here for split tiles).
//
// GB300 design:
//   * One CTA per SM (persistent).  The matrix's blocks (128 rows x 128 k) are
//     dealt out as equal contiguous ranges, one per CTA, so every SM streams
//     the same number of bytes whatever N and K are.  A 128-row tile cut by a
//     range boundary is finished by one statically chosen CTA of those sharing
//     it (the one whose part is expected to end last): the others publish their
//     partial sums as tagged 64-bit words in the workspace, the combiner polls
//     for them (bounded), sums them in CTA order and clears them, so results are
//     deterministic.  Each CTA works on its two cut tiles first, so the fix-up
//     is off the launch's critical tail.
//   * Warp 8 is the producer: one lane issues 1-D bulk copies (TMA engine) of
//     whole stages (4 consecutive blocks of one tile, 33 KB for int4) into a
//     small ring of shared-memory stages tracked by mbarriers (L2 evict-first:
//     every weight byte is read once), and keeps a short window of later stages
//     in flight from HBM into L2 with bulk L2 prefetches.  The CTA of the next
//     launch takes over the SM as soon as this one exits and starts its weight
//     stream before the whole grid has ended.
//   * Warps 0..7 consume: warp w takes rows 64(w&1) .. 64(w&1)+63 of block w>>1
//     of each stage.  Lane l owns two rows of that half; for each 32-k quarter
//     it reads its 16-byte chunk per row (consecutive lanes, conflict-free) and
//     the quarter's activations (same address for all lanes: a broadcast),
//     unpacks int4 (or int6) to int8 lanes with masks and shifts, and runs
//     dp4a.  Per group the int32 dot is exact; the term (d * wscale) * ascale is
//     formed with two fp32 roundings, as in the definition, and accumulated in
//     fp32.
//   * The activations stay in shared memory (as int8 q) for the whole launch.
//     The int8 entry copies q with one bulk copy.  The fused entry reads bf16 x
//     (straight into registers for up to three rows that fit them, else with a
//     bulk copy), takes the per-row amax and quantises it, bit-identical to the
//     standalone kernel.
//   * Programmatic dependent launch: the producer streams weights before the
//     previous kernel in the stream has finished; the activation copy, and every
//     write to y or the workspace, wait for it (griddepcontrol.wait).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "woq_device.cuh"
#include "woq_fastdiv.h"
#include "woq_layout.h"
#include "woq_prologue.cuh"

namespace woq {

struct GemvParams {
  const uint8_t* w;         // packed buffer (header first)
  const void* x;            // bf16 bits [M][K] (bf16 and RMSNorm entries) or fp32 [M][2K] (SwiGLU entry)
  const uint16_t* gamma;    // bf16 bits [K] (RMSNorm entry)
  float eps;                // RMSNorm epsilon
  const int8_t* q;          // int8 [M][K] (int8 entry)
  const float* ascale;      // fp32 [M] (int8 entry)
  float* y;                 // fp32 [M][N]
  uint32_t* status;         // workspace status word
  unsigned long long* parts;  // [ctas][2][M][128] tagged partial sums of split tiles (tag << 32 | fp32 bits)
  uint32_t* sync;           // workspace words of the grid-wide SwiGLU prologue (zero between launches)
  uint16_t* hbuf;           // workspace scratch [M][K] bf16: the SwiGLU prologue's h, one slice per CTA
  int N, K, T, G;
  uint32_t NB;              // T * G blocks; (grid + 1) * NB < 2^32, so partition math stays 32-bit
  FastDiv div_c, div_nb, div_g;  // division by the grid size, NB and G (multiply-high, no divide sequence)
  int stages;               // shared-memory ring stages
  int prefetch_stages;      // stages' worth of weights kept in flight into L2 beyond the ring
  int act_stride;           // bytes between activation rows of q in shared memory (K, or K + 16)
  int act_offset;           // shared-memory offsets (bytes)
  int red_offset;
  int ring_offset;
  int launch_id;            // trace builds only: which trace slot this launch writes
  // The linear that runs after this one (a hint, may be null): once its own weight stream
  // is issued, CTA c brings into L2 the first nx_blocks blocks, in processing order, of the
  // range that CTA c of that launch will stream (its grid nx_C, nx_NB blocks of nx_bb bytes).
  const uint8_t* nx_w;
  uint32_t nx_NB, nx_C, nx_bb, nx_blocks;
  FastDiv nx_div_c, nx_div_g;
  // Bound of the waits on other CTAs of this grid (partner words, SwiGLU arrivals), and a
  // fault to inject for tests of those bounds: 1 = CTA fault_cta never publishes its
  // split-tile partials, 2 = it never counts itself in at the SwiGLU row maxima (0 = none).
  uint64_t wait_ns;
  int fault;
  uint32_t fault_cta;
};

#ifdef WOQ_TRACE
// Trace build only: %globaltimer stamps per (launch slot, CTA, event); no atomics.
constexpr int kTraceSlots = 16;
constexpr int kTraceCtas = 512;
// events: 0..15 phases, 16+s stage s ready (warp 0), 32+i ring load i issued, 48.. combine,
// 56 before the grid wait, 59 / 58 around the split-tile roles, 60..63 prologue phases
constexpr int kTraceEvents = 64;
static __device__ unsigned long long g_trace[kTraceSlots * kTraceCtas * kTraceEvents];
#define WOQ_TRACE_EV(ev)                                                                              \
  do {                                                                                                \
    if (blockIdx.x < kTraceCtas)                                                                      \
      g_trace[((p.launch_id % kTraceSlots) * kTraceCtas + blockIdx.x) * kTraceEvents + (ev)] =        \
          dev::global_timer_ns();                                                                     \
  } while (0)
#define WOQ_TRACE_EV2(ev)                                                                             \
  do {                                                                                                \
    if (blockIdx.x < kTraceCtas)                                                                      \
      g_trace[((launch_id % kTraceSlots) * kTraceCtas + blockIdx.x) * kTraceEvents + (ev)] =          \
          dev::global_timer_ns();                                                                     \
  } while (0)
#else
#define WOQ_TRACE_EV(ev) \
  do {                   \
  } while (0)
#define WOQ_TRACE_EV2(ev) \
  do {                    \
    (void)launch_id;      \
  } while (0)
#endif

namespace kern {

constexpr int kCW = 8;                 // consumer warps: two per block of a stage, 64 rows each
constexpr int kConsumers = kCW * 32;   // 256
constexpr int kSB = 4;                 // blocks per stage
constexpr int kBarConsumers = 1;       // named barrier id for the consumer warps
static_assert(kCW == 2 * kSB, "each block of a stage is split between two consumer warps");

template <int BITS>
struct Fmt {
  static constexpr int kBlockBytes = BITS == 4 ? kBlockBytesW4 : kBlockBytesW6;
  static constexpr float kDotScale = BITS == 4 ? 0.0625f : 0.25f;  // lanes hold 16w (int4) or 4w (int6)
};

// first block of CTA c under an even split of NB blocks over C CTAs ((C + 1) * NB < 2^32)
__device__ __forceinline__ uint32_t range_begin(uint32_t c, uint32_t NB, const FastDiv& C) { return C.div(c * NB); }
// CTA whose range holds block b
__device__ __forceinline__ uint32_t cta_of_block(uint32_t b, const FastDiv& NB, uint32_t C) { return NB.div((b + 1) * C - 1); }

// Expected finish time, in blocks streamed, of CTA c's part of tile t, for a tile that
// CTA c shares (its first or last tile) under the processing order of ItemOrder.
__device__ __forceinline__ uint32_t part_finish(uint32_t c, uint32_t t, uint32_t NB, const FastDiv& C,
                                                const FastDiv& G) {
  const uint32_t bb = range_begin(c, NB, C), be = range_begin(c + 1, NB, C);
  const uint32_t ft = G.div(bb), lt = G.div(be - 1);
  if (ft == lt) return be - bb;
  const uint32_t a = (ft + 1) * G.d - bb;   // the start item, processed first
  return t == ft ? a : a + (be - lt * G.d);  // the end item, processed second
}

// The CTA that combines split tile t, shared by CTAs c_first .. c_last: the one whose part
// is expected to finish last (ties: the lowest CTA).  Every CTA sharing the tile reaches
// the same answer.  Warp-wide: lane k evaluates sharers c_first + k, c_first + k + 32, ...
// and two warp reductions pick the largest finish time, then the lowest CTA holding it.
__device__ __forceinline__ uint32_t combiner_of(uint32_t t, uint32_t c_first, uint32_t c_last, uint32_t NB,
                                                const FastDiv& C, const FastDiv& G, int lane) {
  uint32_t best_f = 0, best_c = 0xFFFFFFFFu;  // a sharer's part holds at least one block: f >= 1
  for (uint32_t base = c_first; base <= c_last; base += 32) {  // warp-uniform
    const uint32_t c2 = base + (uint32_t)lane;
    if (c2 <= c_last) {
      const uint32_t f = part_finish(c2, t, NB, C, G);
      if (f > best_f) {  // a lane visits its sharers in increasing order: ties keep the lowest
        best_f = f;
        best_c = c2;
      }
    }
  }
  const uint32_t f_max = __reduce_max_sync(0xffffffffu, best_f);
  return __reduce_min_sync(0xffffffffu, best_f == f_max ? best_c : 0xFFFFFFFFu);
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

// One half block (rows 64h .. 64h+63 x one group) by one warp:
// acc[jj][m] += term(row 32(2h+jj)+lane, m).  The int4 (or int6) lanes of the low and
// high nibbles accumulate into separate int32 chains (more independent dp4a), summed
// exactly at the end of the group.
template <int BITS, int M, int R, int C>
__device__ __forceinline__ void consume_half_block(const uint8_t* __restrict__ blk, const int8_t* __restrict__ act,
                                                   int qs, int g, int lane, int h, const float (&as)[M],
                                                   float (&acc)[R][C]) {
  static_assert(R >= 2 && C >= M, "accumulators [2][M] (or a wider array)");
  const uint2 sc = *reinterpret_cast<const uint2*>(blk + 8 * lane);
  const uint32_t sw = h ? sc.y : sc.x;  // scales of rows 32(2h) + lane and 32(2h+1) + lane
  float wsc[2];
  wsc[0] = dev::half_bits_to_float(sw & 0xFFFFu) * Fmt<BITS>::kDotScale;
  wsc[1] = dev::half_bits_to_float(sw >> 16) * Fmt<BITS>::kDotScale;

  int dlo[2][M], dhi[2][M];
#pragma unroll
  for (int jj = 0; jj < 2; ++jj)
#pragma unroll
    for (int m = 0; m < M; ++m) dlo[jj][m] = dhi[jj][m] = 0;

  const int8_t* ag = act + g * kGroup;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 v[2];
    uint2 u[2] = {make_uint2(0u, 0u), make_uint2(0u, 0u)};
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int j = 2 * h + jj;
      v[jj] = *reinterpret_cast<const uint4*>(blk + w4_chunk_offset(c, j, lane));
      if constexpr (BITS == 6)
        u[jj] = *reinterpret_cast<const uint2*>(blk + hi_chunk_offset(c, j, lane));
    }
    uint32_t a[M][8];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const uint4 a0 = *reinterpret_cast<const uint4*>(ag + m * qs + 32 * c);
      const uint4 a1 = *reinterpret_cast<const uint4*>(ag + m * qs + 32 * c + 16);
      a[m][0] = a0.x; a[m][1] = a0.y; a[m][2] = a0.z; a[m][3] = a0.w;
      a[m][4] = a1.x; a[m][5] = a1.y; a[m][6] = a1.z; a[m][7] = a1.w;
    }
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const uint32_t vw[4] = {v[jj].x, v[jj].y, v[jj].z, v[jj].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t lo, hi;
        unpack_word<BITS>(vw[i], (i < 2) ? u[jj].x : u[jj].y, i & 1, lo, hi);
#pragma unroll
        for (int m = 0; m < M; ++m) {
          dlo[jj][m] = dev::dp4a_ss(lo, a[m][2 * i], dlo[jj][m]);
          dhi[jj][m] = dev::dp4a_ss(hi, a[m][2 * i + 1], dhi[jj][m]);
        }
      }
    }
  }
#pragma unroll
  for (int jj = 0; jj < 2; ++jj)
#pragma unroll
    for (int m = 0; m < M; ++m) {
      // (d * wscale) * ascale with two fp32 roundings; lanes carry 16d (int4) or 4d (int6),
      // and wsc carries wscale / 16 (or / 4), so the first product is exactly fl(d * wscale)
      const float t = __fmul_rn(__fmul_rn(dev::small_int_to_float(dlo[jj][m] + dhi[jj][m]), wsc[jj]), as[m]);
      acc[jj][m] = __fadd_rn(acc[jj][m], t);
    }
}

// ---------------------------------------------------------------------------------------
// Tensor-core consumer (int4): one half block by one warp with the f16 MMA
// mma.sync m16n8k16 (fp32 accumulate).  Lane L = 4g + t.  The warp's 64 rows are four
// 16-row m-tiles; in m-tile mt lane L supplies rows 16mt + g and 16mt + g + 8, 32-k
// quarter t of the group (one 16-byte chunk per row).  Word i of a chunk (k0 = 32t + 8i)
// feeds two MMAs, one for its low nibbles (k0 .. k0+3), one for its high nibbles
// (k0+4 .. k0+7), with A elements made by a single LOP3 each:
//   low:  f16(1024 + (w + 8))       high: f16(1024 + 16 (w + 8))
// (the nibble's top bit flipped gives w + 8 in [0, 15]).  B is q of activation row g
// (zero for g >= M) at the same k, converted to f16 exactly.  Products and every partial
// sum are integers below 2^24, so the fp32 accumulators are exact whatever order the
// tensor core adds in.  With S_lo and S_hi the sums of q over the group's low- and
// high-nibble positions,
//   d = acc_lo + acc_hi / 16 - (1032 S_lo + 72 S_hi) = sum_k w q
// exactly (every intermediate below 9.2e6 < 2^24).  acc[mt][v] accumulates d * wscale over
// the groups for (row g + 8 (v >> 1), column 2t + (v & 1)) of m-tile mt; the caller
// applies the activation scale.
__device__ __forceinline__ uint32_t lop3_sel_xor(uint32_t a, uint32_t mask, uint32_t c) {
  uint32_t d;  // mask ? a ^ c : c
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(mask), "r"(c));
  return d;
}

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// int8 q bytes (q0, q1, q2, q3) -> f16x2 (q0, q2) and (q1, q3), exact
__device__ __forceinline__ void q4_to_f16x2(uint32_t q4, uint32_t& b02, uint32_t& b13) {
  const uint32_t u = q4 ^ 0x80808080u;  // q + 128 per byte
  uint32_t r02 = __byte_perm(u, 0x64646464u, 0x4240);  // f16 1024 + q + 128
  uint32_t r13 = __byte_perm(u, 0x64646464u, 0x4341);
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(r02) : "r"(0x64806480u));  // - 1152
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(r13) : "r"(0x64806480u));
  b02 = r02;
  b13 = r13;
}

template <int M>
__device__ __forceinline__ void consume_half_block_mma(const uint8_t* __restrict__ blk, const int8_t* __restrict__ act,
                                                       int qs, int g_idx, int lane, int h, float (&acc)[4][4]) {
  const int g = lane >> 2, t = lane & 3;
  // B fragments and the group's offset correction for activation row g
  uint32_t bl0[4], bl1[4], bh0[4], bh1[4];
  int corr = 0;
  if (g < M) {
    const int8_t* ap = act + g * qs + g_idx * kGroup + 32 * t;
    const uint4 qa = *reinterpret_cast<const uint4*>(ap);
    const uint4 qb = *reinterpret_cast<const uint4*>(ap + 16);
    const uint32_t qw[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    int s_lo = 0, s_hi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      q4_to_f16x2(qw[2 * i], bl0[i], bl1[i]);
      q4_to_f16x2(qw[2 * i + 1], bh0[i], bh1[i]);
      s_lo = dev::dp4a_ss(qw[2 * i], 0x01010101u, s_lo);
      s_hi = dev::dp4a_ss(qw[2 * i + 1], 0x01010101u, s_hi);
    }
    corr = 1032 * s_lo + 72 * s_hi;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) bl0[i] = bl1[i] = bh0[i] = bh1[i] = 0u;
  }
  corr += __shfl_xor_sync(0xffffffffu, corr, 1);
  corr += __shfl_xor_sync(0xffffffffu, corr, 2);
  // columns 2t, 2t+1 of D are activation rows 2t, 2t+1: their corrections
  const float c0 = -(float)__shfl_sync(0xffffffffu, corr, 8 * t);
  const float c1 = -(float)__shfl_sync(0xffffffffu, corr, 8 * t + 4);

  // fp16 weight scales of rows 16mt + g + 8s: word [mt & 1][s] holds m-tiles (mt & 1, (mt & 1) + 2)
  // as its (low, high) halves
  uint32_t sw[2][2];
#pragma unroll
  for (int p = 0; p < 2; ++p)
#pragma unroll
    for (int s = 0; s < 2; ++s)
      sw[p][s] = *reinterpret_cast<const uint32_t*>(blk + 2 * (scale_index(16 * p + 8 * s + g) + 2 * h));

  const int gx = g ^ (2 * t);
  // two m-tiles at a time: four independent accumulator chains per warp
#pragma unroll
  for (int mp = 0; mp < 2; ++mp) {
    const uint8_t* base = blk + kScaleBytes + ((4 * t + 2 * h + mp) * 32 + gx) * 16;
    uint32_t wa[2][4], wb[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u) {  // m-tile 2mp + u: rows 16(2mp+u) + g (+8) sit at lane slot 16u + gx (+8)
      const uint4 va = *reinterpret_cast<const uint4*>(base + (16 * u) * 16);
      const uint4 vb = *reinterpret_cast<const uint4*>(base + (16 * u + 8) * 16);
      wa[u][0] = va.x; wa[u][1] = va.y; wa[u][2] = va.z; wa[u][3] = va.w;
      wb[u][0] = vb.x; wb[u][1] = vb.y; wb[u][2] = vb.z; wb[u][3] = vb.w;
    }
    float dl[2][4], dh[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int v = 0; v < 4; ++v) dl[u][v] = dh[u][v] = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t a = wa[u][i], b = wb[u][i], sa = a >> 8, sb = b >> 8;
        mma_16816(dl[u], lop3_sel_xor(a, 0x000F000Fu, 0x64086408u), lop3_sel_xor(b, 0x000F000Fu, 0x64086408u),
                  lop3_sel_xor(sa, 0x000F000Fu, 0x64086408u), lop3_sel_xor(sb, 0x000F000Fu, 0x64086408u), bl0[i],
                  bl1[i]);
        mma_16816(dh[u], lop3_sel_xor(a, 0x00F000F0u, 0x64806480u), lop3_sel_xor(b, 0x00F000F0u, 0x64806480u),
                  lop3_sel_xor(sa, 0x00F000F0u, 0x64806480u), lop3_sel_xor(sb, 0x00F000F0u, 0x64806480u), bh0[i],
                  bh1[i]);
      }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int mt = 2 * mp + u;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        // acc_lo + acc_hi / 16 (<= 9.1e6) and the correction are exact, so d is the exact group dot
        const float d = __fadd_rn(__fmaf_rn(dh[u][v], 0.0625f, dl[u][v]), (v & 1) ? c1 : c0);
        const uint32_t w2 = sw[u][v >> 1];
        const float ws = dev::half_bits_to_float(mp == 0 ? (w2 & 0xFFFFu) : (w2 >> 16));
        acc[mt][v] = __fmaf_rn(d, ws, acc[mt][v]);
      }
    }
  }
}

// The blocks of one CTA's range, as work items (tile t, groups [ga, gb)) in processing
// order: the partial tile at the start of the range, then the partial tile at its
// end, then the whole tiles in between.  Split tiles are thereby finished early, and
// the launch ends on tiles that need no fix-up.
struct ItemOrder {
  uint32_t b_begin, b_end, first_tile, last_tile;
  int G, n_items;
  __device__ __forceinline__ ItemOrder(uint32_t bb, uint32_t be, const FastDiv& g)
      : b_begin(bb), b_end(be), G((int)g.d) {
    first_tile = g.div(bb);
    last_tile = g.div(be - 1);
    n_items = (int)(last_tile - first_tile + 1);
  }
  __device__ __forceinline__ void get(int i, uint32_t& t, int& ga, int& gb) const {
    if (first_tile == last_tile) {
      t = first_tile;
      ga = (int)(b_begin - t * G);
      gb = (int)(b_end - t * G);
    } else if (i == 0) {
      t = first_tile;
      ga = (int)(b_begin - t * G);
      gb = G;
    } else if (i == 1) {
      t = last_tile;
      ga = 0;
      gb = (int)(b_end - t * G);
    } else {
      t = first_tile + (i - 1);
      ga = 0;
      gb = G;
    }
  }
};

// Walks the ring stages (up to kSB consecutive blocks of one item) in processing order.
struct StageCursor {
  const ItemOrder* order;
  int item;
  uint32_t t;
  int ga, gb, g0;
  __device__ __forceinline__ void start(const ItemOrder* o) {
    order = o;
    item = 0;
    order->get(0, t, ga, gb);
    g0 = ga;
  }
  __device__ __forceinline__ bool valid() const { return item < order->n_items; }
  __device__ __forceinline__ int nb() const { return gb - g0 < kSB ? gb - g0 : kSB; }
  __device__ __forceinline__ uint32_t block() const { return t * (uint32_t)order->G + (uint32_t)g0; }
  __device__ __forceinline__ void advance() {
    g0 += kSB;
    if (g0 >= gb) {
      ++item;
      if (item < order->n_items) {
        order->get(item, t, ga, gb);
        g0 = ga;
      }
    }
  }
};

// L2 prefetch of the next linear's weights ("What is the bottleneck?": a decode step is a
// run of weight reads, one linear after another).  A launch leaves the memory idle from
// the moment its last weights have landed until the next launch's CTAs have started and
// issued their own stream; the next launch's first stages are fetched in that gap instead.
// CTA c takes the range CTA c of the next launch will stream (the same even partition) and
// prefetches its first nx_blocks blocks in that launch's processing order (the partial
// tile at the start of the range, the one at its end, then the whole tiles), in pieces of
// at most 32 KiB.  Issued by the producer lane after the last copy of this launch's own
// stream, so these bytes queue behind this launch's.
static __device__ __noinline__ void prefetch_next_linear(const GemvParams& p, uint32_t cta) {
  const uint32_t bb = range_begin(cta, p.nx_NB, p.nx_div_c);
  const uint32_t be = range_begin(cta + 1, p.nx_NB, p.nx_div_c);
  if (be <= bb) return;
  const ItemOrder o(bb, be, p.nx_div_g);
  const uint8_t* blocks = p.nx_w + kHeaderBytes;
  uint32_t left = p.nx_blocks;
  const uint32_t per_piece = (32u * 1024u) / p.nx_bb > 0 ? (32u * 1024u) / p.nx_bb : 1u;
  for (int i = 0; i < o.n_items && left > 0; ++i) {
    uint32_t t;
    int ga, gb;
    o.get(i, t, ga, gb);
    uint32_t b = t * (uint32_t)o.G + (uint32_t)ga;
    uint32_t n = (uint32_t)(gb - ga) < left ? (uint32_t)(gb - ga) : left;
    left -= n;
    while (n > 0) {
      const uint32_t k = n < per_piece ? n : per_piece;
      dev::bulk_prefetch_l2(blocks + (size_t)b * p.nx_bb, k * p.nx_bb);
      b += k;
      n -= k;
    }
  }
}

// Activation prologue of the fused entry, run by the consumer warps on the bf16 x
// that one bulk copy placed at act[0, 2 M K) (or, with X_GLOBAL, on x in global
// memory): per-row amax, scale = amax / 127, and q = rne(x / scale) written to
// act + m qs for row m (qs = K or K + 16 <= 2K, so in place the q byte of value e
// overwrites only x bytes of values with index <= e).
//
// The amax covers the whole row; q is only formed for k in [klo1, khi1) and [klo2, khi2),
// the groups this CTA's blocks read (the rest of the tile is never looked at).
//
// Rows with K <= kConsumers * 8 * (kRegVecs / M) are read once into registers (from
// shared memory, or straight from global memory with X_GLOBAL); the barrier after the
// amax pass then guarantees that every x value has been read before any q byte is
// written.  Longer rows are quantised in rounds, each read in
// full before any thread of the round writes (the amax pass has read everything
// before the first write, so skipped rounds need no reads).  A row's codes come from the
// division-free corrected quotient (quantise8_fast) when its scale allows it (row_fast),
// else from the IEEE division (quantise8_exact); both give rne(fl(x / s)).
constexpr int kRegVecs = 12;  // 8-value vectors per thread kept in registers

// Row scale s = RN(amax / 127) and rc = RN(1 / s) for a bf16 amax held in an fp32, by the
// IEEE division and reciprocal.  An all-zero row gets s = 0 and rc = 0 (quantise8_fast then
// yields q = 0).  (Two constant tables of significands, read after a warm-up load, gave the
// same bits; the step was 0.6 % slower at one row, 1.7 % at four.)
__device__ __forceinline__ void scale_and_rcp(float amax, float& s, float& rc) {
  if (amax == 0.0f) {
    s = 0.0f;
    rc = 0.0f;
  } else {
    s = __fdiv_rn(amax, 127.0f);
    rc = __frcp_rn(s);
  }
}

// Eight bf16 values -> eight q bytes, q = rne(RN(x / s)) without a division, the pairs in
// packed fp32x2 arithmetic (woq_quotient.h): t = RN(x rc), r = RN(x - t s) by a fused
// multiply-add, u = RN(t + r rc) (the correction step of Markstein's division), and
// y = RN(u + 1.5 2^23), whose low byte is rne(u) mod 256.  ns2 holds -s.  rne(u) equals the
// code of the IEEE quotient for every bf16 x with |x| <= amax whenever amax >= 2^-116
// (row_fast); other rows take quantise8_exact.
__device__ __forceinline__ uint2 quantise8_fast(uint4 xv, dev::f32x2 rc2, dev::f32x2 ns2) {
  const dev::f32x2 magic = dev::f2_splat(dev::kRoundMagic);
  const uint32_t w4[4] = {xv.x, xv.y, xv.z, xv.w};
  uint32_t yb[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const dev::f32x2 x = dev::f2_pack(w4[i] << 16, w4[i] & 0xFFFF0000u);  // values 2i, 2i+1
    const dev::f32x2 t = dev::f2_mul(x, rc2);
    const dev::f32x2 r = dev::f2_fma(t, ns2, x);
    const dev::f32x2 u = dev::f2_fma(r, rc2, t);
    const dev::f32x2 y = dev::f2_add(u, magic);
    yb[2 * i] = dev::f2_lo(y);
    yb[2 * i + 1] = dev::f2_hi(y);
  }
  return make_uint2(__byte_perm(__byte_perm(yb[0], yb[1], 0x0040), __byte_perm(yb[2], yb[3], 0x0040), 0x5410),
                    __byte_perm(__byte_perm(yb[4], yb[5], 0x0040), __byte_perm(yb[6], yb[7], 0x0040), 0x5410));
}

// Eight q bytes by the IEEE division, for rows with amax below 2^-116 (none in practice);
// kept out of line so the common path carries no division code.
static __device__ __noinline__ uint2 quantise8_exact(uint4 xv, float sc) {
  const uint32_t w4[4] = {xv.x, xv.y, xv.z, xv.w};
  uint32_t qb[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    qb[i] = dev::quant_byte_exact(__uint_as_float((i & 1) ? (w4[i >> 1] & 0xFFFF0000u) : (w4[i >> 1] << 16)), sc);
  return make_uint2(qb[0] | (qb[1] << 8) | (qb[2] << 16) | (qb[3] << 24),
                    qb[4] | (qb[5] << 8) | (qb[6] << 16) | (qb[7] << 24));
}

// bf16x2 absmax accumulator over one 8-value vector
__device__ __forceinline__ uint32_t absmax8(uint32_t acc, uint4 v) {
  return dev::bf16x2_absmax(acc, dev::bf16x2_absmax(dev::bf16x2_absmax(v.x, v.y), dev::bf16x2_absmax(v.z, v.w)));
}

// Per-row amax partials of this thread -> every thread's row scales and reciprocals
// (one barrier).  s_scratch holds [M rows][8 warps] partials.
template <int M>
__device__ __forceinline__ void row_scales(const float (&lmax)[M], int tid, int lane, int warp, float* s_scratch,
                                           float* s_as, float (&sc)[M], float (&rc)[M]) {
#pragma unroll
  for (int m = 0; m < M; ++m) {
    // non-negative floats order like their bit patterns
    const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(lmax[m]));
    if (lane == 0) s_scratch[m * kCW + warp] = __uint_as_float(wm);
  }
  dev::named_barrier_sync(kBarConsumers, kConsumers);
  if constexpr (M == 1) {
    const float4 a = *reinterpret_cast<const float4*>(s_scratch);
    const float4 b = *reinterpret_cast<const float4*>(s_scratch + 4);
    const float amax = fmaxf(fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)), fmaxf(fmaxf(b.x, b.y), fmaxf(b.z, b.w)));
    scale_and_rcp(amax, sc[0], rc[0]);
    if (tid == 0) s_as[0] = sc[0];
  } else {
    // thread m works out row m (the rows' chains in parallel, not one after another in every
    // thread) and leaves the reciprocal in its row's first scratch slot
    if (tid < M) {
      const float4 a = *reinterpret_cast<const float4*>(s_scratch + tid * kCW);
      const float4 b = *reinterpret_cast<const float4*>(s_scratch + tid * kCW + 4);
      const float amax = fmaxf(fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)), fmaxf(fmaxf(b.x, b.y), fmaxf(b.z, b.w)));
      float s, r;
      scale_and_rcp(amax, s, r);
      s_as[tid] = s;
      s_scratch[tid * kCW] = r;
    }
    dev::named_barrier_sync(kBarConsumers, kConsumers);
#pragma unroll
    for (int m = 0; m < M; ++m) {
      sc[m] = s_as[m];
      rc[m] = s_scratch[m * kCW];
    }
  }
}

// Whether a row's codes come from quantise8_fast: its scale s = RN(amax / 127) is zero (an
// all-zero row: rc = 0 gives u = 0, q = 0) or at least 2^-123, i.e. amax >= 2^-116.  Uniform
// across the row, so a warp never diverges on it.
__device__ __forceinline__ bool row_fast(float s) { return s == 0.0f || s >= 0x1p-123f; }

// Eight q bytes of one vector of a row: the division-free route or, for rows too small for
// it, the IEEE division.
__device__ __forceinline__ uint2 quantise8(uint4 xv, dev::f32x2 rc2, dev::f32x2 ns2, float s, bool fast) {
  return fast ? quantise8_fast(xv, rc2, ns2) : quantise8_exact(xv, s);
}

// X_GLOBAL: rows that fit registers are read straight from x in global memory (L2 only: the
// previous grid wrote them) instead of from a bf16 copy in shared memory; longer rows are not
// taken that way (the caller copies them).
template <int M, bool X_GLOBAL = false>
__device__ __forceinline__ void quantise_prologue(uint8_t* act, int K, int qs, int klo1, int khi1, int klo2, int khi2,
                                                  int tid, int lane, int warp, float* s_scratch, float* s_as,
                                                  int launch_id, const uint16_t* xg = nullptr) {
  constexpr int kVPR = kRegVecs / M;  // vectors per row held in registers
  constexpr int kStride = kConsumers * 8;  // values per vector round of all threads
  const uint16_t* xs = reinterpret_cast<const uint16_t*>(act);
  float sc[M], rc[M];
  if (K <= kStride * kVPR) {
    uint4 xv[M][kVPR];
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
      for (int j = 0; j < kVPR; ++j) {
        const int k = 8 * tid + kStride * j;
        if constexpr (X_GLOBAL)
          xv[m][j] = k < K ? __ldcg(reinterpret_cast<const uint4*>(xg + (size_t)m * K + k)) : make_uint4(0, 0, 0, 0);
        else
          xv[m][j] = k < K ? *reinterpret_cast<const uint4*>(xs + m * K + k) : make_uint4(0, 0, 0, 0);
      }
    float lmax[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      uint32_t acc = 0;
#pragma unroll
      for (int j = 0; j < kVPR; ++j) {
        if (kStride * j >= K) break;  // warp-uniform
        acc = absmax8(acc, xv[m][j]);  // zeros beyond the row
      }
      lmax[m] = dev::bf16x2_absmax_to_float(acc);
    }
    row_scales<M>(lmax, tid, lane, warp, s_scratch, s_as, sc, rc);  // every x value was read before this barrier
    if (tid == 0) WOQ_TRACE_EV2(5);
    dev::f32x2 rc2[M], ns2[M];
    bool fast[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      rc2[m] = dev::f2_splat(rc[m]);
      ns2[m] = dev::f2_splat(-sc[m]);
      fast[m] = row_fast(sc[m]);
    }
    bool all_fast = true;  // CTA-uniform: the division route's call stays out of the common loop
#pragma unroll
    for (int m = 0; m < M; ++m) all_fast = all_fast && fast[m];
    if (all_fast) {
#pragma unroll
      for (int j = 0; j < kVPR; ++j) {
        if (kStride * j >= K) break;  // uniform
        const int k = 8 * tid + kStride * j;
        if (k < K && ((k >= klo1 && k < khi1) || (k >= klo2 && k < khi2))) {  // read by this CTA
#pragma unroll
          for (int m = 0; m < M; ++m)
            *reinterpret_cast<uint2*>(act + m * qs + k) = quantise8_fast(xv[m][j], rc2[m], ns2[m]);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < kVPR; ++j) {
        if (kStride * j >= K) break;  // uniform
        const int k = 8 * tid + kStride * j;
        if (k < K && ((k >= klo1 && k < khi1) || (k >= klo2 && k < khi2))) {
#pragma unroll
          for (int m = 0; m < M; ++m)
            *reinterpret_cast<uint2*>(act + m * qs + k) = quantise8(xv[m][j], rc2[m], ns2[m], sc[m], fast[m]);
        }
      }
    }
    return;
  }
  // longer rows: amax pass, then rounds of 4 vectors per thread over each row
  float lmax[M];
#pragma unroll
  for (int m = 0; m < M; ++m) {
    uint32_t a[4] = {0u, 0u, 0u, 0u};
    int k = 8 * tid;
    for (; k + 3 * kStride < K; k += 4 * kStride) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        a[u] = absmax8(a[u], *reinterpret_cast<const uint4*>(xs + m * K + k + u * kStride));
    }
    for (; k < K; k += kStride) a[0] = absmax8(a[0], *reinterpret_cast<const uint4*>(xs + m * K + k));
    lmax[m] = dev::bf16x2_absmax_to_float(dev::bf16x2_absmax(dev::bf16x2_absmax(a[0], a[1]),
                                                             dev::bf16x2_absmax(a[2], a[3])));
  }
  row_scales<M>(lmax, tid, lane, warp, s_scratch, s_as, sc, rc);
  if (tid == 0) WOQ_TRACE_EV2(5);
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const dev::f32x2 rc2 = dev::f2_splat(rc[m]);
    const dev::f32x2 ns2 = dev::f2_splat(-sc[m]);
    const bool fast = row_fast(sc[m]);  // CTA-uniform: the division route's call stays out of the common loop
    for (int k0 = 0; k0 < K; k0 += 4 * kStride) {
      // CTA-uniform: skip rounds that hold no k this CTA reads
      if (!((k0 < khi1 && k0 + 4 * kStride > klo1) || (k0 < khi2 && k0 + 4 * kStride > klo2))) continue;
      uint4 xv[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const int k = k0 + 8 * tid + kStride * v;
        xv[v] = k < K ? *reinterpret_cast<const uint4*>(xs + m * K + k) : make_uint4(0, 0, 0, 0);
      }
      dev::named_barrier_sync(kBarConsumers, kConsumers);
      if (fast) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int k = k0 + 8 * tid + kStride * v;
          if (k < K && ((k >= klo1 && k < khi1) || (k >= klo2 && k < khi2)))
            *reinterpret_cast<uint2*>(act + m * qs + k) = quantise8_fast(xv[v], rc2, ns2);
        }
      } else {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int k = k0 + 8 * tid + kStride * v;
          if (k < K && ((k >= klo1 && k < khi1) || (k >= klo2 && k < khi2)))
            *reinterpret_cast<uint2*>(act + m * qs + k) = quantise8_exact(xv[v], sc[m]);
        }
      }
    }
  }
}

// Prologue of a kernel instance: what the launch receives as activations.
//   kProInt8:   int8 q [M][K] and fp32 scales [M] (act_quant run before);
//   kProBf16:   bf16 x [M][K], quantised by the consumer warps (the fused entry);
//   kProRms:    bf16 x [M][K] and bf16 gamma [K]: RMSNorm, then quantisation;
//   kProSwiglu: the fp32 [M][2K] output of a gate+up linear: SwiGLU, then quantisation.
enum Prologue { kProInt8 = 0, kProBf16 = 1, kProRms = 2, kProSwiglu = 3 };

// RMSNorm of the bf16 rows at act (landed by the bulk copy), in place, by the consumer
// warps (see woq_prologue.cuh for the definition).  s_bits[M]: row max |x| bits, s_sum[M]:
// integer sums of squares, both zero on entry; shared-memory atomics make both
// independent of the order the warps arrive in.
template <int M>
__device__ __forceinline__ void rmsnorm_prologue(uint8_t* act, int K, const uint16_t* __restrict__ gamma, float eps,
                                                 int tid, int lane, uint32_t* s_bits, unsigned long long* s_sum) {
  constexpr int kStride = kConsumers * 8;
  uint16_t* xs = reinterpret_cast<uint16_t*>(act);
#pragma unroll
  for (int m = 0; m < M; ++m) {
    uint32_t acc = 0;
    for (int k = 8 * tid; k < K; k += kStride) acc = absmax8(acc, *reinterpret_cast<const uint4*>(xs + m * K + k));
    const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(dev::bf16x2_absmax_to_float(acc)));
    if (lane == 0) atomicMax(s_bits + m, wm);
  }
  dev::named_barrier_sync(kBarConsumers, kConsumers);
  int C[M];
#pragma unroll
  for (int m = 0; m < M; ++m) {
    C[m] = pro::rms_row_exponent(s_bits[m]);
    unsigned long long part = 0;
    if (C[m] != -1000) {
      for (int k = 8 * tid; k < K; k += kStride) {
        const uint4 v = *reinterpret_cast<const uint4*>(xs + m * K + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) part += pro::rms_term(w[i] & 0xFFFFu, C[m]) + pro::rms_term(w[i] >> 16, C[m]);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0 && part) atomicAdd(s_sum + m, part);
  }
  dev::named_barrier_sync(kBarConsumers, kConsumers);  // every x read before the first h write
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const float r = C[m] == -1000 ? 0.0f : pro::rms_rcp(s_sum[m], C[m], K, eps);
    for (int k = 8 * tid; k < K; k += kStride) {
      uint4* px = reinterpret_cast<uint4*>(xs + m * K + k);
      *px = pro::rms_h8(*px, __ldg(reinterpret_cast<const uint4*>(gamma + k)), r);
    }
  }
  dev::named_barrier_sync(kBarConsumers, kConsumers);
}

// RMSNorm and quantisation of rows held in registers (K <= kRmsRegVecs * 2048, M <= 4):
// the same steps and arithmetic as rmsnorm_prologue followed by quantise_prologue (row
// exponent, exact integer sum of squares, r, h = bf16(RN(RN(x r) gamma)), the row's largest
// |h|, q for the CTA's k ranges), with x read from shared memory once, gamma already in
// registers (loaded before the grid wait: it is a weight) and h never written back.
// s_bits: [0, M) row max |x| bits, [8, 8 + M) row max |h| bits, zero on entry; s_part:
// [M][8 warps] sums of squares, written before they are read.
constexpr int kRmsRegVecs = 3;
template <int M>
__device__ __forceinline__ void rmsnorm_quantise_regs(uint8_t* act, int K, int qs, const uint4 (&gv)[kRmsRegVecs],
                                                      float eps, int klo1, int khi1, int klo2, int khi2, int tid,
                                                      int lane, uint32_t* s_bits, unsigned long long* s_part,
                                                      float* s_as, int launch_id) {
  constexpr int kStride = kConsumers * 8;
  const uint16_t* xs = reinterpret_cast<const uint16_t*>(act);
  if (tid == 0) WOQ_TRACE_EV2(60);
  uint4 v[M][kRmsRegVecs];
#pragma unroll
  for (int m = 0; m < M; ++m)
#pragma unroll
    for (int j = 0; j < kRmsRegVecs; ++j) {
      const int k = 8 * tid + kStride * j;
      v[m][j] = k < K ? *reinterpret_cast<const uint4*>(xs + m * K + k) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
  for (int m = 0; m < M; ++m) {
    uint32_t acc = 0;
#pragma unroll
    for (int j = 0; j < kRmsRegVecs; ++j) acc = absmax8(acc, v[m][j]);
    const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(dev::bf16x2_absmax_to_float(acc)));
    if (lane == 0 && wm) atomicMax(s_bits + m, wm);
  }
  dev::named_barrier_sync(kBarConsumers, kConsumers);  // also: every x value read before any q byte is written
  if (tid == 0) WOQ_TRACE_EV2(61);
  int C[M];
#pragma unroll
  for (int m = 0; m < M; ++m) {
    C[m] = pro::rms_row_exponent(s_bits[m]);
    unsigned long long part = 0;
    if (C[m] != -1000) {
#pragma unroll
      for (int j = 0; j < kRmsRegVecs; ++j) {  // zero vectors beyond the row add nothing
        const uint32_t w[4] = {v[m][j].x, v[m][j].y, v[m][j].z, v[m][j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) part += pro::rms_term(w[i] & 0xFFFFu, C[m]) + pro::rms_term(w[i] >> 16, C[m]);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) s_part[m * 8 + (tid >> 5)] = part;  // one slot per warp: no atomics
  }
  dev::named_barrier_sync(kBarConsumers, kConsumers);
  if (tid == 0) WOQ_TRACE_EV2(62);
#pragma unroll
  for (int m = 0; m < M; ++m) {
    unsigned long long S = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) S += s_part[m * 8 + w];  // integer: any order gives the same sum
    const float r = C[m] == -1000 ? 0.0f : pro::rms_rcp(S, C[m], K, eps);
    uint32_t acc = 0;
#pragma unroll
    for (int j = 0; j < kRmsRegVecs; ++j) {
      if (8 * tid + kStride * j < K) {
        v[m][j] = pro::rms_h8(v[m][j], gv[j], r);
        acc = absmax8(acc, v[m][j]);
      }
    }
    const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(dev::bf16x2_absmax_to_float(acc)));
    if (lane == 0 && wm) atomicMax(s_bits + 8 + m, wm);
  }
  dev::named_barrier_sync(kBarConsumers, kConsumers);
  if (tid == 0) WOQ_TRACE_EV2(63);
#pragma unroll
  for (int m = 0; m < M; ++m) {
    float sc, rc;
    scale_and_rcp(__uint_as_float(s_bits[8 + m]), sc, rc);
    if (tid == 0) s_as[m] = sc;
    const dev::f32x2 rc2 = dev::f2_splat(rc);
    const dev::f32x2 ns2 = dev::f2_splat(-sc);
    if (row_fast(sc)) {  // CTA-uniform: the division route's call stays out of the common loop
#pragma unroll
      for (int j = 0; j < kRmsRegVecs; ++j) {
        const int k = 8 * tid + kStride * j;
        if (k < K && ((k >= klo1 && k < khi1) || (k >= klo2 && k < khi2)))
          *reinterpret_cast<uint2*>(act + m * qs + k) = quantise8_fast(v[m][j], rc2, ns2);
      }
    } else {
#pragma unroll
      for (int j = 0; j < kRmsRegVecs; ++j) {
        const int k = 8 * tid + kStride * j;
        if (k < K && ((k >= klo1 && k < khi1) || (k >= klo2 && k < khi2)))
          *reinterpret_cast<uint2*>(act + m * qs + k) = quantise8_exact(v[m][j], sc);
      }
    }
  }
}

// Fused SwiGLU prologue, split over the grid.  h = SwiGLU(gate, up) of the fp32 [M][2K]
// rows at gu (see woq_prologue.cuh).  The quantisation needs the largest |h| of each whole
// row, and a CTA reads the k ranges of its own blocks, which many CTAs share.  So each CTA of
// the first half of the grid forms h once for its part of each row, stores it (bf16) in the
// workspace scratch rows, folds its largest |h| into the row words with red.max (|h| as bits
// orders like the values; the result does not depend on the order) and counts itself in
// with a release reduction; once all of them have (every CTA of this grid is resident, the
// wait is bounded) every CTA reads the row maxima and the h of its own ranges and quantises
// them like a bf16 activation.  sync (workspace, zero between launches): [0] arrivals, [2] departures
// (CTAs that have read the maxima), [8 + m] row m's largest |h| bits; CTA 0 zeroes them at
// the end of the launch (swiglu_sync_reset).
template <int M>
__device__ __forceinline__ void swiglu_grid_max(uint32_t* sync, uint32_t C, const uint32_t (&acc)[M], int tid,
                                                int lane, float* s_scratch, volatile int* s_ok, uint64_t wait_ns,
                                                bool skip_arrival, int launch_id) {
  uint32_t* s_max = reinterpret_cast<uint32_t*>(s_scratch);  // [M] this CTA's largest |h| bits
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(dev::bf16x2_absmax_to_float(acc[m])));
    if (lane == 0 && wm) atomicMax(s_max + m, wm);
  }
  dev::named_barrier_sync(kBarConsumers, kConsumers);
  if (tid == 0) {
    WOQ_TRACE_EV2(61);
    for (int m = 0; m < M; ++m)
      if (s_max[m]) dev::red_max_relaxed_u32(sync + 8 + m, s_max[m]);
    if (!skip_arrival) dev::red_add_release_u32(sync, 1u);  // ordered after the maxima
    bool ok = true;
    const uint64_t t0 = dev::global_timer_ns();
    while (dev::ld_acquire_u32(sync) < C) {  // one poller per CTA, backed off so the arrivals get through
      if (dev::global_timer_ns() - t0 > wait_ns) {
        ok = false;
        break;
      }
      __nanosleep(32);
    }
    for (int m = 0; m < M; ++m) s_scratch[8 + m] = __uint_as_float(ok ? dev::ld_acquire_u32(sync + 8 + m) : 0u);
    if (ok) dev::red_add_release_u32(sync + 2, 1u);  // after the reads above
    *s_ok = ok ? 1 : 0;
    WOQ_TRACE_EV2(62);
  }
  dev::named_barrier_sync(kBarConsumers, kConsumers);
}

// Returns 0 if the wait ran out, 1 once q of this CTA's k ranges is in the activation area.
template <int M>
__device__ __forceinline__ int swiglu_split_prologue(uint8_t* act, int K, int qs, const float* __restrict__ gu,
                                                     uint32_t* sync, uint16_t* hbuf, uint32_t cta, uint32_t C,
                                                     int klo1, int khi1, int klo2, int khi2, int tid, int lane,
                                                     int warp, float* s_scratch, float* s_as, volatile int* s_ok,
                                                     uint64_t wait_ns, bool skip_arrival, int launch_id) {
  uint32_t* s_max = reinterpret_cast<uint32_t*>(s_scratch);
  if (tid < M) s_max[tid] = 0u;
  dev::named_barrier_sync(kBarConsumers, kConsumers);
  if (tid == 0) WOQ_TRACE_EV2(60);
  // This CTA's slice of every row: h once, into the scratch rows, one value per consumer
  // thread and pass (a slice is a few hundred values, so every thread takes part and the
  // exp / reciprocal chain runs once per value rather than eight times in a row).  Only the first half of the
  // grid forms slices: CTAs are placed in index order, and the last ones often start only
  // when the previous grid ends, so the row maxima do not wait for them.
  const uint32_t Cw = (C + 1) / 2;  // CTAs that form a slice
  const int n_lo = cta < Cw ? (int)((unsigned long long)cta * (unsigned)K / Cw) : 0;
  const int n_hi = cta < Cw ? (int)((unsigned long long)(cta + 1) * (unsigned)K / Cw) : 0;
  uint32_t acc[M];
#pragma unroll
  for (int m = 0; m < M; ++m) {
    acc[m] = 0u;
    for (int k = n_lo + tid; k < n_hi; k += kConsumers) {
      const uint32_t h = pro::swiglu_bf16(__ldg(gu + (size_t)m * 2 * K + k), __ldg(gu + (size_t)m * 2 * K + K + k));
      hbuf[(size_t)m * K + k] = (uint16_t)h;
      acc[m] = dev::bf16x2_absmax(acc[m], h);
    }
  }
  // also publishes the slices; only the CTAs that formed one count themselves in
  swiglu_grid_max<M>(sync, Cw, acc, tid, lane, s_scratch, s_ok, wait_ns, skip_arrival || cta >= Cw, launch_id);
  if (!*s_ok) return 0;
  float sc[M];
  dev::f32x2 rc2[M], ns2[M];
  bool fast[M];
#pragma unroll
  for (int m = 0; m < M; ++m) {
    float rc;
    scale_and_rcp(s_scratch[8 + m], sc[m], rc);
    rc2[m] = dev::f2_splat(rc);
    ns2[m] = dev::f2_splat(-sc[m]);
    fast[m] = row_fast(sc[m]);
  }
#pragma unroll
  for (int m = 0; m < M; ++m)
    if (tid == m) s_as[m] = sc[m];
  // h of the k ranges this CTA's blocks read, written by the CTAs that own those slices,
  // read through L2 (this SM's L1 may hold an older launch's lines) and quantised straight
  // into the activation area: per batch up to kHB vectors of 8 values per row and thread,
  // every load issued before the first is used, so a batch costs one round trip (one batch
  // covers the 27B down projection's ranges at M <= 4)
  constexpr int kHB = M <= 2 ? 4 : (M <= 4 ? 3 : 1);
  const int nv1 = (khi1 - klo1) / 8, nv2 = (khi2 - klo2) / 8;
  const int per_row = nv1 + nv2;
  for (int v0 = tid; v0 < per_row; v0 += kHB * kConsumers) {
    uint4 hv[M][kHB];
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
      for (int b = 0; b < kHB; ++b) {
        const int v = v0 + b * kConsumers;
        if (v < per_row) {
          const int k = v < nv1 ? klo1 + 8 * v : klo2 + 8 * (v - nv1);
          hv[m][b] = __ldcg(reinterpret_cast<const uint4*>(hbuf + (size_t)m * K + k));
        }
      }
#pragma unroll
    for (int m = 0; m < M; ++m) {
      if (fast[m]) {  // CTA-uniform: the division route's call stays out of the common loop
#pragma unroll
        for (int b = 0; b < kHB; ++b) {
          const int v = v0 + b * kConsumers;
          if (v < per_row) {
            const int k = v < nv1 ? klo1 + 8 * v : klo2 + 8 * (v - nv1);
            *reinterpret_cast<uint2*>(act + m * qs + k) = quantise8_fast(hv[m][b], rc2[m], ns2[m]);
          }
        }
      } else {
#pragma unroll
        for (int b = 0; b < kHB; ++b) {
          const int v = v0 + b * kConsumers;
          if (v < per_row) {
            const int k = v < nv1 ? klo1 + 8 * v : klo2 + 8 * (v - nv1);
            *reinterpret_cast<uint2*>(act + m * qs + k) = quantise8_exact(hv[m][b], sc[m]);
          }
        }
      }
    }
  }
  return 1;
}

// End of a launch with the split SwiGLU prologue: CTA 0 waits (bounded) until every CTA
// has read the row maxima, then zeroes the words for the next launch.  false on timeout.
template <int M>
__device__ __forceinline__ bool swiglu_sync_reset(uint32_t* sync, uint32_t C, uint64_t wait_ns) {
  const uint64_t t0 = dev::global_timer_ns();
  while (dev::ld_acquire_u32(sync + 2) < C)
    if (dev::global_timer_ns() - t0 > wait_ns) return false;
  sync[0] = 0u;
  sync[2] = 0u;
#pragma unroll
  for (int m = 0; m < M; ++m) sync[8 + m] = 0u;
  return true;
}

// Consumer of a kernel instance: every consumer warp on dp4a, or every one on the f16
// tensor-core MMA.
enum Consumer { kDp4a = 0, kMma = 1 };

template <int BITS, int M, int PRO, int CONS>
// One CTA per SM: the nine warps put three on one sub-partition, whose 16,384 registers then
// allow 168 per thread (3 x 32 x 168 = 16,128).  The cap was 112; at 168 the kernels use what
// they need (114 at one row, 140 at four) and the 27B step got 0.2 % (M = 1) to 1.4 % (M = 3)
// faster.  80, which let two CTAs share an SM, spilled and was slower (M = 1 2.47 against
// 2.33 ms); 96 without spills let the next launch's CTA share the SM and was slower too (M = 1
// 2.37 against 2.31 ms, M = 3 4.34 against 3.19): the next launch's ring fill then competes
// with this launch's own stream.
__global__ void __maxnreg__(168) gemv_kernel(const GemvParams p) {
  constexpr bool FUSED = PRO != kProInt8;  // activations quantised inside this launch
  static_assert(CONS == kDp4a || BITS == 4, "the tensor-core consumer reads int4 blocks");
  static_assert(CONS == kMma || M <= kMaxMDp4a, "dp4a kernels take up to four activation rows");
  constexpr int BB = Fmt<BITS>::kBlockBytes;
  constexpr int kStageBytes = kSB * BB;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);          // [8]
  uint64_t* empty = full + 8;                                  // [8]
  uint64_t* actbar = full + 16;                                // activations landed
  volatile int* s_flags = reinterpret_cast<volatile int*>(smem + 136);  // [0] ticket-last, [1] abort, [2] header-ok, [3] prologue barrier ok
  float* s_as = reinterpret_cast<float*>(smem + 160);          // [M] activation scales
  float* s_scratch = reinterpret_cast<float*>(smem + 192);     // [8 rows][8 warps] amax partials, to byte 448
  unsigned long long* s_sum = reinterpret_cast<unsigned long long*>(smem + 448);  // [8] RMSNorm sums of squares
  unsigned long long* s_part = reinterpret_cast<unsigned long long*>(smem + 512);  // [8 rows][8 warps] of them
  uint8_t* act = smem + p.act_offset;                          // bf16 x, quantised in place (fused) or int8 q
  float* red = reinterpret_cast<float*>(smem + p.red_offset);  // [4 blocks][M][128 rows]
  uint8_t* ring = smem + p.ring_offset;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t C = gridDim.x;
  const uint32_t cta = blockIdx.x;
  const uint32_t b_begin = range_begin(cta, p.NB, p.div_c);
  const uint32_t b_end = range_begin(cta + 1, p.NB, p.div_c);
  const int G = p.G;
  const int stages = p.stages;
  const ItemOrder order(b_begin, b_end, p.div_g);

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      dev::mbar_init(full + s, 1);
      dev::mbar_init(empty + s, kCW);
    }
    dev::mbar_init(actbar, 1);
    s_flags[0] = 0;
    s_flags[1] = 0;
    s_flags[2] = 1;
    dev::fence_mbar_init();
  }
  if constexpr (PRO == kProRms) {
    if (tid < 16) reinterpret_cast<uint32_t*>(s_scratch)[tid] = 0u;
    if (tid < 8) s_sum[tid] = 0ull;
  }
  __syncthreads();
  if (tid == 0) WOQ_TRACE_EV(0);
  // every CTA of this grid is resident (one per SM), so the next grid may be scheduled now
  dev::pdl_launch_dependents();

  if (warp == kCW) {
    // ---------------------------------------------------------------- producer
    // weights do not depend on the previous grid: no griddepcontrol.wait here
    if (lane == 0) {
      const uint64_t pol = dev::l2_evict_first_policy();
      const uint8_t* blocks = p.w + kHeaderBytes;
      StageCursor ld, pf;
      ld.start(&order);
      long long it = 0;
      bool ok = true;
      for (; ld.valid() && it < stages; ld.advance(), ++it) {
        const int slot = (int)it;
        const uint32_t bytes = (uint32_t)(ld.nb() * BB);
        dev::mbar_arrive_expect_tx(full + slot, bytes);
        dev::bulk_copy_g2s(ring + (size_t)slot * kStageBytes, blocks + (size_t)ld.block() * BB, bytes, full + slot, pol);
        if (it < 16) WOQ_TRACE_EV(32 + (int)it);
      }
      WOQ_TRACE_EV(1);
      // keep prefetch_stages stages beyond the ring in flight into L2
      pf = ld;
      for (int k = 0; k < p.prefetch_stages && pf.valid(); ++k, pf.advance())
        dev::bulk_prefetch_l2(blocks + (size_t)pf.block() * BB, (uint32_t)(pf.nb() * BB));
      int slot = 0;
      uint32_t phase = 0;  // parity of the empty-barrier phase to wait for
      for (; ld.valid(); ld.advance(), ++it) {
        if (!dev::mbar_wait_bounded(empty + slot, phase)) {
          ok = false;
          break;
        }
        // consumers that gave up release slots without waiting for them to land: issue
        // nothing more into the ring (the flag is written before any such release)
        if (s_flags[1]) break;
        const uint32_t bytes = (uint32_t)(ld.nb() * BB);
        dev::mbar_arrive_expect_tx(full + slot, bytes);
        dev::bulk_copy_g2s(ring + (size_t)slot * kStageBytes, blocks + (size_t)ld.block() * BB, bytes, full + slot, pol);
        if (it < 16) WOQ_TRACE_EV(32 + (int)it);
        if (pf.valid()) {
          dev::bulk_prefetch_l2(blocks + (size_t)pf.block() * BB, (uint32_t)(pf.nb() * BB));
          pf.advance();
        }
        if (++slot == stages) {
          slot = 0;
          phase ^= 1u;
        }
      }
      WOQ_TRACE_EV(9);
      if (ok && p.nx_w != nullptr && cta < p.nx_C) prefetch_next_linear(p, cta);
      if (!ok) atomicOr(p.status, 0x2u /* WOQ_DEVERR_TIMEOUT */);
      // no bulk copy may still be landing in this CTA's shared memory when it exits
      dev::mbar_wait_bounded(actbar, 0);
      const long long first = it > stages ? it - stages : 0;
      for (long long i = first; i < it; ++i) dev::mbar_wait_bounded(full + (int)(i % stages), (uint32_t)((i / stages) & 1));
      WOQ_TRACE_EV(2);
    }
    return;
  }

  // -------------------------------------------------------------------- consumers
  if (tid == 0) WOQ_TRACE_EV(59);
  // roles in the split tiles (only the first two items can be split), worked out while the
  // previous grid may still be running
  // (per split item: whether this CTA combines it, the first and last CTA sharing the tile,
  // and which part slot the first of them publishes it in; a later sharer starts its range
  // inside the tile, so the tile is its first part)
  bool comb0 = false, comb1 = false;
  uint32_t cf0 = 0, cl0 = 0, cf1 = 0, cl1 = 0;
  int fp0 = 0, fp1 = 0;
  {
    uint32_t t;
    int ga, gb;
    order.get(0, t, ga, gb);
    if (!(ga == 0 && gb == G)) {
      cf0 = cta_of_block(t * G, p.div_nb, C);
      cl0 = cta_of_block(t * G + G - 1, p.div_nb, C);
      comb0 = combiner_of(t, cf0, cl0, p.NB, p.div_c, p.div_g, lane) == cta;
      fp0 = range_begin(cf0, p.NB, p.div_c) < t * (uint32_t)G ? 1 : 0;
    }
    if (order.n_items > 1) {
      order.get(1, t, ga, gb);
      if (!(ga == 0 && gb == G)) {
        cf1 = cta_of_block(t * G, p.div_nb, C);
        cl1 = cta_of_block(t * G + G - 1, p.div_nb, C);
        comb1 = combiner_of(t, cf1, cl1, p.NB, p.div_c, p.div_g, lane) == cta;
        fp1 = range_begin(cf1, p.NB, p.div_c) < t * (uint32_t)G ? 1 : 0;
      }
    }
  }
  if (tid == 0) WOQ_TRACE_EV(58);
  // k ranges of the activations this CTA's blocks read: the start item's groups [ga, G) of
  // its first tile and, for a range that ends in a second tile, [0, gb) of that tile; with
  // whole tiles in between, everything
  int klo1 = 0, khi1 = p.K, klo2 = 0, khi2 = 0;
  {
    uint32_t t;
    int ga, gb;
    order.get(0, t, ga, gb);
    if (order.n_items == 1) {
      klo1 = ga * kGroup;
      khi1 = gb * kGroup;
    } else if (order.n_items == 2) {
      int ga1, gb1;
      order.get(1, t, ga1, gb1);
      if (gb1 < ga) {
        klo1 = 0;
        khi1 = gb1 * kGroup;
        klo2 = ga * kGroup;
        khi2 = p.K;
      }
    }
  }
  // RMSNorm rows that fit registers: gamma (a weight) is loaded before the grid wait
  constexpr bool kRmsRegPath = PRO == kProRms && M <= 4;
  const bool rms_regs = kRmsRegPath && p.K <= kConsumers * 8 * kRmsRegVecs;
  uint4 gv[kRmsRegVecs];
  if constexpr (kRmsRegPath) {
#pragma unroll
    for (int j = 0; j < kRmsRegVecs; ++j) {
      const int k = 8 * tid + kConsumers * 8 * j;
      gv[j] = rms_regs && k < p.K ? __ldg(reinterpret_cast<const uint4*>(p.gamma + k)) : make_uint4(0, 0, 0, 0);
    }
  }
  // the packed header (weights: not written by the previous grid) is fetched before the wait;
  // the ring never reads it, so it would cost a DRAM round trip on the critical path
  uint4 hdr0 = make_uint4(0, 0, 0, 0), hdr1 = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    hdr0 = __ldg(reinterpret_cast<const uint4*>(p.w));
    hdr1 = __ldg(reinterpret_cast<const uint4*>(p.w + 16));
  }
  if (tid == 0) WOQ_TRACE_EV(56);
  // bf16 rows that fit registers are read by the consumers themselves after the grid wait (no
  // bulk copy and mbarrier round trip on the launch's critical path).  27B step: M = 1 2.337 ->
  // 2.309 ms, M = 2 2.731 -> 2.703, M = 3 3.214 -> 3.200; M = 4 went the other way (3.663 ->
  // 3.726) and keeps the bulk copy.
  constexpr bool kXDirect = PRO == kProBf16 && M <= 3;
  const bool x_direct = kXDirect && p.K <= kConsumers * 8 * (kRegVecs / M);
  // activations (and y, the workspace) belong to the previous grid until it has completed
  dev::pdl_wait_prior_grids();
  if (tid == 0) {
    WOQ_TRACE_EV(3);
    const uint32_t act_bytes = (uint32_t)(FUSED ? 2 * M * p.K : M * p.K);
    if (PRO == kProSwiglu || x_direct) {
      dev::mbar_arrive(actbar);  // nothing to copy: the consumers read the rows themselves
    } else if (FUSED || p.act_stride == p.K) {
      dev::mbar_arrive_expect_tx(actbar, act_bytes);
      dev::bulk_copy_g2s(act, FUSED ? p.x : static_cast<const void*>(p.q), act_bytes, actbar);
    } else {
      dev::mbar_arrive_expect_tx(actbar, act_bytes);
      for (int m = 0; m < M; ++m)
        dev::bulk_copy_g2s(act + m * p.act_stride, p.q + (size_t)m * p.K, (uint32_t)p.K, actbar);
    }
  }
  float ascale_in = 0.0f;
  if (!FUSED && tid < M) ascale_in = p.ascale[tid];

  bool aborted = false;
  if (!dev::mbar_wait_bounded(actbar, 0)) {
    aborted = true;
    s_flags[1] = 1;
    atomicOr(p.status, 0x2u /* WOQ_DEVERR_TIMEOUT */);
  }
  if (tid == 0) {
    WOQ_TRACE_EV(4);
    // the packed header must describe this call's (bits, N, K)
    const bool hok = hdr0.x == kMagic && hdr0.y == kLayoutVersion && hdr0.z == (uint32_t)BITS &&
                     hdr0.w == (uint32_t)kTileRows && hdr1.x == (uint32_t)p.N && hdr1.y == (uint32_t)p.K;
    if (!hok) {
      s_flags[2] = 0;
      atomicOr(p.status, 0x1u /* WOQ_DEVERR_HEADER */);
    }
  }
  bool quantised = false;
  if constexpr (kRmsRegPath) {
    if (rms_regs) {
      rmsnorm_quantise_regs<M>(act, p.K, p.act_stride, gv, p.eps, klo1, khi1, klo2, khi2, tid, lane,
                               reinterpret_cast<uint32_t*>(s_scratch), s_part, s_as, p.launch_id);
      quantised = true;
    }
  }
  if constexpr (PRO == kProRms)
    if (!quantised) rmsnorm_prologue<M>(act, p.K, p.gamma, p.eps, tid, lane, reinterpret_cast<uint32_t*>(s_scratch), s_sum);
  if constexpr (PRO == kProSwiglu) {
    const int route = swiglu_split_prologue<M>(act, p.K, p.act_stride, static_cast<const float*>(p.x), p.sync,
                                               p.hbuf, cta, C, klo1, khi1, klo2, khi2, tid, lane, warp, s_scratch,
                                               s_as, s_flags + 3, p.wait_ns, p.fault == 2 && cta == p.fault_cta,
                                               p.launch_id);
    if (tid == 0) WOQ_TRACE_EV(63);
    if (route == 0) {
      aborted = true;
      if (tid == 0) {
        s_flags[1] = 1;
        atomicOr(p.status, 0x2u /* WOQ_DEVERR_TIMEOUT */);
      }
    }
  } else if constexpr (PRO == kProBf16) {
    if (kXDirect && x_direct)
      quantise_prologue<M, kXDirect>(act, p.K, p.act_stride, klo1, khi1, klo2, khi2, tid, lane, warp, s_scratch, s_as,
                                 p.launch_id, static_cast<const uint16_t*>(p.x));
    else
      quantise_prologue<M>(act, p.K, p.act_stride, klo1, khi1, klo2, khi2, tid, lane, warp, s_scratch, s_as,
                           p.launch_id);
  } else if constexpr (FUSED) {
    if (!quantised)
      quantise_prologue<M>(act, p.K, p.act_stride, klo1, khi1, klo2, khi2, tid, lane, warp, s_scratch, s_as,
                           p.launch_id);
  } else {
    if (tid < M) s_as[tid] = ascale_in;
  }
  dev::named_barrier_sync(kBarConsumers, kConsumers);
  if (tid == 0) WOQ_TRACE_EV(6);

  const int8_t* actq = reinterpret_cast<const int8_t*>(act);
  float as[M];
#pragma unroll
  for (int m = 0; m < M; ++m) as[m] = s_as[m];
  const bool header_ok = s_flags[2] != 0;
  const int hb = warp >> 1;  // block of the stage this warp works on
  const int hh = warp & 1;   // its row half

  int slot = 0;
  uint32_t phase = 0;  // parity of the full-barrier phase to wait for
  bool first_stage = true;
#ifdef WOQ_TRACE
  int n_stage = 0;
#endif
  for (int item = 0; item < order.n_items; ++item) {
    uint32_t t;
    int ga, gb;
    order.get(item, t, ga, gb);

    // dp4a: [row half][m]; MMA: [m-tile][fragment]
    constexpr int kAccR = CONS == kDp4a ? 2 : 4, kAccC = CONS == kDp4a ? M : 4;
    float acc[kAccR][kAccC];
#pragma unroll
    for (int jj = 0; jj < kAccR; ++jj)
#pragma unroll
      for (int m = 0; m < kAccC; ++m) acc[jj][m] = 0.0f;

    for (int g0 = ga; g0 < gb; g0 += kSB) {
      const int nb = gb - g0 < kSB ? gb - g0 : kSB;
      // (the outcome is made warp-uniform: the tensor-core consumer shuffles across the warp)
      if (!aborted && !__all_sync(0xffffffffu, dev::mbar_wait_bounded(full + slot, phase))) {
        aborted = true;
        s_flags[1] = 1;
        atomicOr(p.status, 0x2u /* WOQ_DEVERR_TIMEOUT */);
      }
      if (tid == 0 && first_stage) WOQ_TRACE_EV(7);
      first_stage = false;
#ifdef WOQ_TRACE
      if (tid == 0 && n_stage < 16) WOQ_TRACE_EV(16 + n_stage);
      ++n_stage;
#endif
      if (!aborted && hb < nb) {
        const uint8_t* blk = ring + (size_t)slot * kStageBytes + (size_t)hb * BB;
        if constexpr (CONS == kDp4a) {
          consume_half_block<BITS, M>(blk, actq, p.act_stride, g0 + hb, lane, hh, as, acc);
        } else {
          consume_half_block_mma<M>(blk, actq, p.act_stride, g0 + hb, lane, hh, acc);
        }
      }
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(empty + slot);
      if (++slot == stages) {
        slot = 0;
        phase ^= 1u;
      }
    }

    // reduce the four blocks' partial sums for this tile: red[block][m][row]
    if constexpr (CONS == kMma) {
      // MMA sums are sum_g d * wscale; the activation scale of columns 2t, 2t+1 is applied here
      const int g = lane >> 2, t2 = 2 * (lane & 3);
      const float a0 = s_as[t2 < M ? t2 : M - 1], a1 = s_as[t2 + 1 < M ? t2 + 1 : M - 1];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int m = t2 + (v & 1);
          if (m < M)
            red[(hb * M + m) * kTileRows + 64 * hh + 16 * mt + g + 8 * (v >> 1)] =
                __fmul_rn(acc[mt][v], (v & 1) ? a1 : a0);
        }
    } else {
#pragma unroll
      for (int jj = 0; jj < 2; ++jj)
#pragma unroll
        for (int m = 0; m < M; ++m) red[(hb * M + m) * kTileRows + 64 * hh + 32 * jj + lane] = acc[jj][m];
    }
    dev::named_barrier_sync(kBarConsumers, kConsumers);
    const bool write_ok = header_ok && s_flags[1] == 0;
    const int row = tid & (kTileRows - 1);
    const bool row_thread = tid < kTileRows;
    const uint32_t n = t * kTileRows + row;
    float sum[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float s = red[(0 * M + m) * kTileRows + row];
#pragma unroll
      for (int b = 1; b < kSB; ++b) s = __fadd_rn(s, red[(b * M + m) * kTileRows + row]);
      sum[m] = s;
    }
    dev::named_barrier_sync(kBarConsumers, kConsumers);  // red may be rewritten from here on
    if (tid == 0 && item == 0) WOQ_TRACE_EV(10);
    if (tid == 0 && item == 1) WOQ_TRACE_EV(11);
    if (ga == 0 && gb == G) {
      if (write_ok && row_thread && n < p.N) {
#pragma unroll
        for (int m = 0; m < M; ++m) p.y[(size_t)m * p.N + n] = sum[m];
      }
    } else {
      // Tile split across CTAs.  The part expected to finish last (its CTA is the
      // "combiner") sums all parts in CTA order and writes y; every other CTA publishes its
      // part as tagged 64-bit words (value and tag land in one store, so a reader that sees
      // the tag sees the value) and moves on.  No atomics, no barrier: the combiner polls
      // (bounded) and clears the words for the next launch.
      if (row_thread) {
        const uint32_t c_first = item == 0 ? cf0 : cf1;
        const uint32_t c_last = item == 0 ? cl0 : cl1;
        const int first_part = item == 0 ? fp0 : fp1;
        const bool comb = item == 0 ? comb0 : comb1;
        if (!comb) {
          if (write_ok && !(p.fault == 1 && cta == p.fault_cta)) {
            const int part = (t == order.first_tile) ? 0 : 1;
            unsigned long long* mine = p.parts + ((size_t)(cta * 2 + part) * M) * kTileRows;
#pragma unroll
            for (int m = 0; m < M; ++m)
              dev::st_relaxed_u64(mine + m * kTileRows + row, (1ull << 32) | __float_as_uint(sum[m]));
          }
        } else if (write_ok) {
          if (tid == 0) WOQ_TRACE_EV(12 + (item == 0 ? 0 : 2));
          // issue the loads of up to kBatch partner parts at once (one round trip), then poll
          // only the words that were not there yet; sum in CTA order
          constexpr int kBatch = M == 1 ? 8 : (M == 2 ? 4 : (M <= 4 ? 2 : 1));  // bounded by registers
          float tot[M];
#pragma unroll
          for (int m = 0; m < M; ++m) tot[m] = 0.0f;
          bool ok = true;
          for (uint32_t cb = c_first; cb <= c_last; cb += kBatch) {
            unsigned long long w[kBatch][M];
            unsigned long long* src[kBatch];
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
              const uint32_t c2 = cb + b;
              src[b] = nullptr;
              if (c2 <= c_last && c2 != cta) {
                const int part2 = c2 == c_first ? first_part : 0;
                src[b] = p.parts + ((size_t)(c2 * 2 + part2) * M) * kTileRows + row;
#pragma unroll
                for (int m = 0; m < M; ++m) w[b][m] = dev::ld_relaxed_u64(src[b] + m * kTileRows);
              }
            }
            if (tid == 0 && cb == c_first) WOQ_TRACE_EV(48 + (item == 0 ? 0 : 2));
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
              const uint32_t c2 = cb + b;
              if (c2 > c_last) break;
              if (c2 == cta) {
#pragma unroll
                for (int m = 0; m < M; ++m) tot[m] = __fadd_rn(tot[m], sum[m]);
                continue;
              }
#pragma unroll
              for (int m = 0; m < M; ++m) {
                unsigned long long v = w[b][m];
                if (!(v >> 32)) {
                  const uint64_t t0 = dev::global_timer_ns();
                  while (!(v >> 32)) {
                    if (dev::global_timer_ns() - t0 > p.wait_ns) break;
                    __nanosleep(16);
                    v = dev::ld_relaxed_u64(src[b] + m * kTileRows);
                  }
                }
                if (!(v >> 32)) ok = false;
                if (tid == 0 && cb == c_first) WOQ_TRACE_EV(49 + (item == 0 ? 0 : 2));
                tot[m] = __fadd_rn(tot[m], __uint_as_float((uint32_t)v));
                dev::st_relaxed_u64(src[b] + m * kTileRows, 0ull);  // ready for the next launch
              }
            }
          }
          if (tid == 0) WOQ_TRACE_EV(13 + (item == 0 ? 0 : 2));
          if (!ok) {
            atomicOr(p.status, 0x2u /* WOQ_DEVERR_TIMEOUT */);
          } else if (n < p.N) {
#pragma unroll
            for (int m = 0; m < M; ++m) p.y[(size_t)m * p.N + n] = tot[m];
          }
        }
      }
    }
  }
  if constexpr (PRO == kProSwiglu) {
    if (cta == 0 && tid == 0 && s_flags[3] && !swiglu_sync_reset<M>(p.sync, C, p.wait_ns))
      atomicOr(p.status, 0x2u /* WOQ_DEVERR_TIMEOUT */);
  }
  if (tid == 0) WOQ_TRACE_EV(8);
}

}  // namespace kern
}  // namespace woq
