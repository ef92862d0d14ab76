// Packed device layout of the weight-only-quantised skinny linear.
//
// Section "Optimizing the Linear Kernel" of "Doubling LLM token rates in
// ComfyUI": the GEMV reads weights and group scales from one buffer laid out in
// its reading order, so each thread block streams a single contiguous run rather
// than two separate tensors.
//
// This file fixes that order for the GB300 kernels:
//
//   [256-byte header][block (tile 0, group 0)][block (0, 1)] ... [block (T-1, G-1)]
//
// T = ceil(N / 128) row tiles, G = K / 128 groups, blocks tile-major, so one
// tile (128 rows x all of K) is one contiguous run and a CTA's share of the
// matrix is a contiguous byte range.
//
// A block covers rows 128t .. 128t+127 and k = 128g .. 128g+127.  Inside it,
// row r is written r = 32j + l (j = 0..3, l = 0..31): consumer lane l of a warp
// owns rows l, 32+l, 64+l, 96+l.
//
//   bytes [0, 256)     fp16 scales; row 32j+l at half-word index 4l + j, so lane
//                      l reads its four scales with one 8-byte load.
//   bytes [256, 8448)  int4 weights: 16 chunks (c, j), c = 0..3 the 32-k quarter
//                      of the group, each chunk 32 lanes x 16 bytes, lane l at
//                      byte 16 (l ^ 2c).  The swizzle keeps both consumer patterns
//                      free of shared-memory bank conflicts: 32 consecutive rows of
//                      one quarter (the dp4a path), and rows {g, g+8} x quarters
//                      {0..3} (the tensor-core path, lane 4g + t reading quarter t).
//                      The 16 bytes of (c, j, l) hold row 32j+l, k = 32c .. 32c+31
//                      as four 32-bit words; word i holds k0 = 32c + 8i .. k0+7:
//                      byte b has k0+b in its low nibble and k0+4+b in its high
//                      nibble (two's complement nibbles).  So (v << 4) & 0xF0F0F0F0
//                      gives 16 * w[k0 .. k0+3] and v & 0xF0F0F0F0 gives
//                      16 * w[k0+4 .. k0+7] as four int8 lanes each.
//   int6 only:
//   bytes [8448, 12544) high two bits of the int6 weights: 16 chunks (c, j) of
//                      32 lanes x 8 bytes.  The low four bits of each int6 weight
//                      (w & 15) sit in the int4 region above, in the same nibble
//                      positions.  The 8 bytes of (c, j, l) are two words u0, u1;
//                      u_h serves int4-region words i = 2h, 2h+1: byte b of u_h
//                      holds, in bits 2s .. 2s+1, the top two bits (w >> 4) & 3 of
//                      the weight k0(i) + b (s = 2(i-2h)) and k0(i) + 4 + b
//                      (s = 2(i-2h) + 1).
//
// Rows beyond N hold zero weights and zero scales.
#pragma once

#include <stddef.h>
#include <stdint.h>

#if defined(__CUDACC__)
#define WOQ_HD __host__ __device__
#else
#define WOQ_HD
#endif

namespace woq {

constexpr uint32_t kMagic = 0x31514F57u;  // "WOQ1" little-endian
constexpr uint32_t kLayoutVersion = 2;
constexpr int kHeaderBytes = 256;
constexpr int kTileRows = 128;
constexpr int kGroup = 128;
constexpr int kScaleBytes = kTileRows * 2;                 // 256
constexpr int kW4Bytes = kTileRows * kGroup / 2;           // 8192
constexpr int kHiBytes = kTileRows * kGroup / 4;           // 4096 (2 bits per weight)
constexpr int kBlockBytesW4 = kScaleBytes + kW4Bytes;      // 8448
constexpr int kBlockBytesW6 = kScaleBytes + kW4Bytes + kHiBytes;  // 12544
constexpr int kMaxM = 8;      // activation rows (int4); int6 and the dp4a kernels take up to kMaxMDp4a
constexpr int kMaxMDp4a = 4;
constexpr long kMaxMK = 98304;  // shared-memory bound on M * K for the activation tile

// Header (little-endian, 256 bytes; unused bytes zero).
struct PackedHeader {
  uint32_t magic;
  uint32_t version;
  uint32_t bits;
  uint32_t tile_rows;
  uint32_t N;
  uint32_t K;
  uint32_t tiles;
  uint32_t groups;
  uint64_t block_bytes;
  uint64_t total_bytes;
};
static_assert(sizeof(PackedHeader) <= kHeaderBytes, "header too large");

WOQ_HD inline int block_bytes(int bits) { return bits == 4 ? kBlockBytesW4 : kBlockBytesW6; }

inline size_t packed_bytes(int bits, long N, long K) {
  if ((bits != 4 && bits != 6) || N < 0 || K < 0 || K % kGroup != 0 || N > 0x7fffffff || K > 0x7fffffff) return 0;
  const size_t tiles = (size_t)((N + kTileRows - 1) / kTileRows);
  const size_t groups = (size_t)(K / kGroup);
  return (size_t)kHeaderBytes + tiles * groups * (size_t)block_bytes(bits);
}

// Byte offset, inside a block, of the 16-byte int4 chunk of quarter c, row group j, lane l.
WOQ_HD inline constexpr int w4_chunk_offset(int c, int j, int l) {
  return kScaleBytes + ((c * 4 + j) * 32 + (l ^ (2 * c))) * 16;
}
// Byte offset, inside a block, of the 8-byte high-bit chunk of quarter c, row group j, lane l (int6).
WOQ_HD inline constexpr int hi_chunk_offset(int c, int j, int l) { return kScaleBytes + kW4Bytes + ((c * 4 + j) * 32 + l) * 8; }
// Half-word index, inside a block's scale area, of row r.
WOQ_HD inline constexpr int scale_index(int r) { return (r % 32) * 4 + r / 32; }

}  // namespace woq
