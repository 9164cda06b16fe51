// The tiled weight layout and the activation records of the mma.sync matmul.
//
// Tiled weights.  Rows form 16-row blocks rb; 16 consecutive blocks form a row group
// (256 rows; the last group may hold fewer blocks, nrb).  Inside a row group the data is
// ordered [64-input chunk c][block in group][...], so the K-range of a whole row group is
// one contiguous byte range (one bulk copy per pipeline stage).  Per (rb, c):
//   words  u32 [32 lanes][4]; lane = 4*gid + tig; word j holds row
//          16*rb + gid + 8*(j&1) of group g = 2c + (j>>1).  Its nibble at bit 4p + 16h
//          (p = 0..3, h = 0..1) carries the code of input 32g + 8p + 2*tig + h, stored as
//          code + 8 (0..15).
//   scales fp16 [8 gid][4] in the same (row, group) order as the words.
// With x a word, the masks x & 0x000F000F, x & 0x00F000F0, (x>>8) & 0x000F000F and
// (x>>8) & 0x00F000F0 are four f16x2 registers of m16n8k16 A fragments: the nibble n at
// bits 0..3 (or 16..19) of a half is the subnormal f16 n * 2^-24, at bits 4..7 it is
// 16n * 2^-24.  Pairs p = 1, 3 carry the extra factor 16, which the activation side
// cancels by holding a/16 for those inputs.
//
// Activation records.  For NT 8-token tiles (NT = 1 for up to 8 tokens, 2 up to 16, 4 up to 32, 8 up to 64) the
// record of chunk c is NT * 1152 bytes at offset c * NT * 1152:
//   [nt][group 0..1][lane] uint4 {h2(a_k, a_k+1), h2(a_k+8, a_k+9)/16,
//                                h2(a_k+16, a_k+17), h2(a_k+24, a_k+25)/16},
//        k = 32g + 2*tig, token 8*nt + gid (f16; a/16 is exact for an int8 a);
//   [group 0..1][nt][tig] float4 {c(t0), c(t0+1), c(t0), c(t0+1)}, t0 = 8*nt + 2*tig,
//        c(t) = -8 * 2^-24 * sum_{k in group} a_k(t), the zero-point correction that seeds
//        the accumulator: sum (q+8) a 2^-24 - 8 sum a 2^-24 = sum q a 2^-24.
// Tokens at or beyond the token count and inputs at or beyond K are zero.
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

// activation records: 8-token tiles for M tokens (1, 2, 4 or 8 tiles: up to 64 tokens), bytes
// per chunk, buffer bytes for K inputs (act_bytes: up to 16 tokens; act_bytes_nt: NT tiles)
__host__ __device__ inline int act_tiles(int M) { return M > 32 ? 8 : (M > 16 ? 4 : (M > 8 ? 2 : 1)); }
__host__ __device__ inline int act_rec_bytes(int NT) { return NT * 1152; }
__host__ __device__ inline size_t act_bytes(int K) { return (size_t)chunks_of(K) * 2 * 1152; }
__host__ __device__ inline size_t act_bytes_nt(int K, int NT) { return (size_t)chunks_of(K) * NT * 1152; }

}  // namespace w4a8
