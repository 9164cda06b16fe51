// The tiled weight layout and the activation fragment layout of the mma.sync matmul.
//
// Tiled weights.  Rows form 16-row blocks rb; 16 consecutive blocks form a row group
// (256 rows; the last group may hold fewer blocks, nrb).  Inside a row group the data is
// ordered [64-input chunk c][block in group][...], so the K-range of a whole row group is
// one contiguous byte range (one bulk copy per pipeline stage).  Per (rb, c):
//   words  u32 [32 lanes][4]; lane = 4*gid + tig; word j holds row
//          16*rb + gid + 8*(j&1) of group 2c + (j>>1); its byte b carries the code of
//          input 32g + 4*tig + b in the low nibble and of input 32g + 16 + 4*tig + b in
//          the high nibble, each stored as code + 8 (0..15).
//   scales fp16 [8 gid][4] in the same (row, group) order as the words.
// Masking a word with 0x0F0F0F0F (or shifting by 4 first) yields the four e4m3 bytes of
// one m16n8k32 A-fragment register: the byte value n in 0..15 is the e4m3 encoding of
// n * 2^-9 (subnormal below 8), so the MMA sees (q + 8) * 2^-9 exactly.
//
// Activation fragments (layout [8-token tile nt][padded group g][lane]): uint4
//   {hi(k0..k0+3), hi(k0+16..k0+19), lo(k0..k0+3), lo(k0+16..k0+19)}, k0 = 32g + 4*tig,
//   token = 8*nt + gid, where an int8 a = 16*hi + lo and the bytes are e4m3 of 16*hi and
//   of lo (exact).  corr[g][token] = -2^-6 * sum_{k in g} a (= -8 * sum a * 2^-9), the
//   negated zero-point correction: sum (q+8) a - 8 sum a = sum q a.
#pragma once
#include <cstddef>

namespace w4a8 {

__host__ __device__ inline int chunks_of(int K) { return (K + 63) / 64; }
__host__ __device__ inline int groups_padded(int K) { return 2 * chunks_of(K); }
__host__ __device__ inline size_t tiled_words(int N, int K) { return (size_t)(N / 16) * chunks_of(K) * 128; }
__host__ __device__ inline size_t tiled_scales(int N, int K) { return (size_t)(N / 16) * chunks_of(K) * 32; }

constexpr int kGroupBlocks = 16;  // 16-row blocks per row group

// Index of the (rb, c) tile among all tiles of an N-row matrix (unit: one tile =
// 128 words = 32 scales).
__host__ __device__ inline size_t tile_index(int N, int KC, int rb, int c) {
  const int n16 = N / 16;
  const int grp = rb / kGroupBlocks, rbl = rb % kGroupBlocks;
  const int nrb = (n16 - grp * kGroupBlocks) < kGroupBlocks ? (n16 - grp * kGroupBlocks) : kGroupBlocks;
  return (size_t)grp * kGroupBlocks * KC + (size_t)c * nrb + rbl;
}

// activation fragment buffer (uint4 units) and correction floats for K inputs
__host__ __device__ inline size_t afrag_uint4(int K) { return (size_t)groups_padded(K) * 2 * 32; }
__host__ __device__ inline size_t corr_floats(int K) { return (size_t)groups_padded(K) * 16; }

}  // namespace w4a8
