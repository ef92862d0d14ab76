// Host packer: canonical checkpoint layout -> interleaved device layout, and back.
//
// Section "Optimizing the Linear Kernel" ("Doubling LLM token rates in
// ComfyUI"): the weights and their group scales are re-laid out once per model
// load into the order the GEMV kernel consumes them.  The byte order is
// defined in woq_layout.h; this file only moves nibbles and half-words.
#include <string.h>

#include "woq.h"
#include "woq_internal.h"
#include "woq_layout.h"

namespace woq {

// canonical 4-bit code of weight (n, k): the raw nibble, two's complement
static inline uint8_t canon_w4_code(const uint8_t* q4, size_t row_bytes, int n, int k) {
  const uint8_t b = q4[(size_t)n * row_bytes + (size_t)(k >> 1)];
  return (k & 1) ? (uint8_t)(b >> 4) : (uint8_t)(b & 0xF);
}

// canonical 6-bit code of weight (n, k)
static inline uint8_t canon_w6_code(const uint8_t* q6, size_t row_bytes, int n, int k) {
  const uint8_t* p = q6 + (size_t)n * row_bytes + (size_t)(k >> 2) * 3;
  const uint32_t word = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16);
  return (uint8_t)((word >> (6 * (k & 3))) & 0x3F);
}

void write_header(void* dst, int bits, int N, int K) {
  PackedHeader h;
  memset(&h, 0, sizeof(h));
  h.magic = kMagic;
  h.version = kLayoutVersion;
  h.bits = (uint32_t)bits;
  h.tile_rows = kTileRows;
  h.N = (uint32_t)N;
  h.K = (uint32_t)K;
  h.tiles = (uint32_t)((N + kTileRows - 1) / kTileRows);
  h.groups = (uint32_t)(K / kGroup);
  h.block_bytes = (uint64_t)block_bytes(bits);
  h.total_bytes = (uint64_t)packed_bytes(bits, N, K);
  memset(dst, 0, kHeaderBytes);
  memcpy(dst, &h, sizeof(h));
}

bool header_matches(const void* src, int bits, int N, int K) {
  PackedHeader h;
  memcpy(&h, src, sizeof(h));
  return h.magic == kMagic && h.version == kLayoutVersion && h.bits == (uint32_t)bits &&
         h.tile_rows == (uint32_t)kTileRows && h.N == (uint32_t)N && h.K == (uint32_t)K &&
         h.total_bytes == (uint64_t)packed_bytes(bits, N, K);
}

static int pack_host(int bits, const uint8_t* q, const uint16_t* scales, int N, int K, void* dst, size_t dst_bytes) {
  const size_t need = packed_bytes(bits, N, K);
  if (need == 0) return WOQ_ERR_SHAPE;
  if (dst == nullptr) return WOQ_ERR_NULL;
  if ((q == nullptr || scales == nullptr) && (size_t)N * (size_t)K > 0) return WOQ_ERR_NULL;
  if (dst_bytes < need) return WOQ_ERR_LAYOUT;
  const int T = (N + kTileRows - 1) / kTileRows;
  const int G = K / kGroup;
  const size_t row_bytes = bits == 4 ? (size_t)K / 2 : (size_t)K / 4 * 3;
  const int bb = block_bytes(bits);
  uint8_t* out = (uint8_t*)dst;
  write_header(out, bits, N, K);
  for (int t = 0; t < T; ++t) {
    for (int g = 0; g < G; ++g) {
      uint8_t* blk = out + kHeaderBytes + ((size_t)t * G + g) * (size_t)bb;
      memset(blk, 0, (size_t)bb);
      uint16_t* sc = (uint16_t*)blk;
      for (int r = 0; r < kTileRows; ++r) {
        const int n = t * kTileRows + r;
        if (n < N) sc[scale_index(r)] = scales[(size_t)n * G + g];
      }
      for (int c = 0; c < 4; ++c)
        for (int j = 0; j < 4; ++j)
          for (int l = 0; l < 32; ++l) {
            const int n = t * kTileRows + 32 * j + l;
            if (n >= N) continue;
            uint8_t* lo = blk + w4_chunk_offset(c, j, l);
            uint8_t* hi = blk + hi_chunk_offset(c, j, l);
            for (int i = 0; i < 4; ++i) {
              const int k0 = g * kGroup + 32 * c + 8 * i;
              for (int b = 0; b < 4; ++b) {
                const uint8_t code_a = bits == 4 ? canon_w4_code(q, row_bytes, n, k0 + b)
                                                 : canon_w6_code(q, row_bytes, n, k0 + b);
                const uint8_t code_b = bits == 4 ? canon_w4_code(q, row_bytes, n, k0 + 4 + b)
                                                 : canon_w6_code(q, row_bytes, n, k0 + 4 + b);
                lo[4 * i + b] = (uint8_t)((code_a & 0xF) | ((code_b & 0xF) << 4));
                if (bits == 6) {
                  const int h = i >> 1, e = i & 1;
                  uint8_t* ub = hi + 4 * h + b;
                  *ub |= (uint8_t)(((code_a >> 4) & 3) << (2 * (2 * e)));
                  *ub |= (uint8_t)(((code_b >> 4) & 3) << (2 * (2 * e + 1)));
                }
              }
            }
          }
    }
  }
  return WOQ_OK;
}

static int unpack_host(int bits, const void* packed, size_t packed_bytes_, int N, int K, uint8_t* q,
                       uint16_t* scales) {
  const size_t need = packed_bytes(bits, N, K);
  if (need == 0) return WOQ_ERR_SHAPE;
  if (packed == nullptr) return WOQ_ERR_NULL;
  if ((q == nullptr || scales == nullptr) && (size_t)N * (size_t)K > 0) return WOQ_ERR_NULL;
  if (packed_bytes_ < need || !header_matches(packed, bits, N, K)) return WOQ_ERR_LAYOUT;
  const int G = K / kGroup;
  const size_t row_bytes = bits == 4 ? (size_t)K / 2 : (size_t)K / 4 * 3;
  const int bb = block_bytes(bits);
  const uint8_t* in = (const uint8_t*)packed;
  if ((size_t)N * row_bytes) memset(q, 0, (size_t)N * row_bytes);
  for (int n = 0; n < N; ++n) {
    const int t = n / kTileRows, r = n % kTileRows, j = r / 32, l = r % 32;
    for (int g = 0; g < G; ++g) {
      const uint8_t* blk = in + kHeaderBytes + ((size_t)t * G + g) * (size_t)bb;
      uint16_t s;
      memcpy(&s, blk + 2 * scale_index(r), 2);
      scales[(size_t)n * G + g] = s;
      for (int c = 0; c < 4; ++c) {
        const uint8_t* lo = blk + w4_chunk_offset(c, j, l);
        const uint8_t* hi = blk + hi_chunk_offset(c, j, l);
        for (int i = 0; i < 4; ++i)
          for (int b = 0; b < 4; ++b)
            for (int half = 0; half < 2; ++half) {
              const int k = g * kGroup + 32 * c + 8 * i + 4 * half + b;
              uint8_t code = half ? (uint8_t)(lo[4 * i + b] >> 4) : (uint8_t)(lo[4 * i + b] & 0xF);
              if (bits == 4) {
                uint8_t* dstb = q + (size_t)n * row_bytes + (size_t)(k >> 1);
                *dstb |= (k & 1) ? (uint8_t)(code << 4) : code;
              } else {
                const int h = i >> 1, e = i & 1;
                const int s2 = 2 * (2 * e + half);
                code |= (uint8_t)(((hi[4 * h + b] >> s2) & 3) << 4);
                uint8_t* p = q + (size_t)n * row_bytes + (size_t)(k >> 2) * 3;
                uint32_t word = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16);
                word |= (uint32_t)code << (6 * (k & 3));
                p[0] = (uint8_t)word;
                p[1] = (uint8_t)(word >> 8);
                p[2] = (uint8_t)(word >> 16);
              }
            }
      }
    }
  }
  return WOQ_OK;
}

}  // namespace woq

extern "C" {

size_t woq_packed_bytes(int bits, int N, int K) { return woq::packed_bytes(bits, N, K); }

int woq_pack_w4(const uint8_t* q4, const uint16_t* scales_f16, int N, int K, void* dst, size_t dst_bytes) {
  return woq::pack_host(4, q4, scales_f16, N, K, dst, dst_bytes);
}

int woq_pack_w6(const uint8_t* q6, const uint16_t* scales_f16, int N, int K, void* dst, size_t dst_bytes) {
  return woq::pack_host(6, q6, scales_f16, N, K, dst, dst_bytes);
}

int woq_unpack(int bits, const void* packed, size_t packed_bytes, int N, int K, uint8_t* q, uint16_t* scales_f16) {
  return woq::unpack_host(bits, packed, packed_bytes, N, K, q, scales_f16);
}

}  // extern "C"
