// Internal interface of the W4A8 mma.sync matmul (shared by the C ABI and the decoder).
#pragma once
#include "common.cuh"
#include "layout.cuh"

namespace w4a8 {

// Fixed schedule of one (K, N) shape.  Every field depends on K and N only, so the
// fp32 reduction order (and hence the bits of y) is the same for every token count.
struct MatmulPlan {
  int N, K;
  int KC;        // 64-input chunks
  int S;         // K slices
  int cps;       // chunks per slice
  int n_rg;      // CTA row groups (kRowsPerCta rows each)
  size_t part_floats;  // split-K partial buffer (S > 1), [S][N][16]
};

constexpr int kWarpsPerCta = 8;
constexpr int kRowBlocksPerWarp = 2;
constexpr int kRowsPerCta = 16 * kWarpsPerCta * kRowBlocksPerWarp;  // 256

MatmulPlan mm_plan(int K, int N);

// Token rows of the EPI_PARTIAL layout (the widest token count a decoder pass uses: a prefill
// bucket of 64 prompt tokens).
constexpr int kPartTokens = 64;
// floats of the EPI_PARTIAL output of a plan: [S][kPartTokens][N]
inline size_t mm_partial_floats(const MatmulPlan& p) { return (size_t)p.S * kPartTokens * p.N; }

// Output handling after the fixed-order reduction: y = fold * s_a[t], then
enum MatmulEpilogue : int {
  EPI_STORE = 0,    // y[t][n] = value
  EPI_ADD = 1,      // y[t][n] += value (residual stream)
  EPI_PARTIAL = 2,  // part[(s * kPartTokens + t) * N + n] = slice s's unscaled sum, t < M; y unused.  The
                    // consumer folds the slices with mm_fold4 / mm_fold2 (no tickets, no fence)
  EPI_ATOMIC = 3,   // y[t][n] += slice value * s_a[t] with a float atomic (y zeroed before): the slices
                    // combine in arrival order -- not deterministic (the fast variant)
};

// Launches the matmul kernel on prepared activation records.  part/tickets: split-K
// scratch (part_floats floats, n_rg counters that must be zero on entry; the kernel
// leaves them zero).
// Raises the dynamic shared-memory limit of the matmul kernels (call once per device,
// outside stream capture).
cudaError_t mm_configure();

// err: device word that receives FLAG_ERR_TIMEOUT if a bounded pipeline wait expires.
// stop: optional device control word; when it has a FLAG_STOP_MASK bit set at kernel
// start (after the dependency wait) the kernel does nothing.
// act: activation records of M tokens (layout.cuh), act_bytes(K) bytes.
cudaError_t mm_run(const MatmulPlan& p, const uint32_t* wt, const uint16_t* st, const uint8_t* act, const float* a_s,
                   int M, float* y, int ldy, int epi, float* part, unsigned* tickets, unsigned* err,
                   const unsigned* stop, cudaStream_t stream);

// Four consecutive outputs (t, n .. n+3) (n % 4 == 0) of an EPI_PARTIAL matmul with S slices
// and N rows: the slices folded left in ascending order and scaled, the same operations (and
// bits) as the kernel's own fold and store.  Every slice's float4 is loaded before the sums
// (8 in flight).
__device__ __forceinline__ float4 mm_fold4(const float* part, int S, int N, int t, int n, const float* a_s) {
  float4 f = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int sb = 0; sb < S; sb += 8) {
    float4 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (sb + q < S) v[q] = *reinterpret_cast<const float4*>(part + ((size_t)(sb + q) * kPartTokens + t) * N + n);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (sb + q >= S) break;
      if (sb + q == 0) {
        f = v[q];
      } else {
        f.x = f.x + v[q].x; f.y = f.y + v[q].y; f.z = f.z + v[q].z; f.w = f.w + v[q].w;
      }
    }
  }
  const float sc = 16777216.0f * a_s[t];
  return make_float4(f.x * sc, f.y * sc, f.z * sc, f.w * sc);
}
// Two outputs (t, n0) and (t, n1), same fold as mm_fold4, loads of both issued together.
__device__ __forceinline__ float2 mm_fold2(const float* part, int S, int N, int t, int n0, int n1, const float* a_s) {
  float f0 = 0.0f, f1 = 0.0f;
  for (int sb = 0; sb < S; sb += 16) {
    float v0[16], v1[16];
#pragma unroll
    for (int q = 0; q < 16; ++q)
      if (sb + q < S) {
        v0[q] = part[((size_t)(sb + q) * kPartTokens + t) * N + n0];
        v1[q] = part[((size_t)(sb + q) * kPartTokens + t) * N + n1];
      }
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      if (sb + q >= S) break;
      f0 = (sb + q == 0) ? v0[q] : f0 + v0[q];
      f1 = (sb + q == 0) ? v1[q] : f1 + v1[q];
    }
  }
  const float sc = 16777216.0f * a_s[t];
  return make_float2(f0 * sc, f1 * sc);
}

// P2 layout (rows [0, N)) -> rows [row0, row0 + N) of an Ntot-row tiled matrix (quant.cu).
cudaError_t repack_run(const uint32_t* w_p2, const uint16_t* s_p2, int N, int K, int Ntot, int row0, uint32_t* w_t,
                       uint16_t* s_t, cudaStream_t st);

// Launches the record builder for int8 activations a_q[M][K] (row stride lda) and zeroes
// n_tickets counters.
cudaError_t act_prep_run(const int8_t* a_q, int M, int K, int lda, uint8_t* act, unsigned* tickets, int n_tickets,
                         cudaStream_t stream, const float* s32 = nullptr);

// Device helpers for fused producers of the activation records (layout.cuh), for M tokens
// (NT = act_tiles(M) tiles).
// act_store_quad: token t (< 8 * NT), inputs k0..k0+3 (k0 % 4 == 0), int8 codes in `codes`
// (byte b = input k0+b): writes the two f16x2 words that hold them.
__device__ __forceinline__ void act_store_quad(uint8_t* act, int NT, int t, int k0, uint32_t codes) {
  const int g = k0 >> 5, kin = k0 & 31;
  const int p = kin >> 3;             // f16x2 word of the fragment (inputs 8p .. 8p+7 of the group)
  const int tig0 = (kin & 7) >> 1;    // 0 or 2: the quad spans lanes tig0 and tig0 + 1
  const float sc = (p & 1) ? 0.0625f : 1.0f;
  const int nt = t >> 3, gid = t & 7;
  uint8_t* frag = act + (size_t)(g >> 1) * act_rec_bytes(NT) + (nt * 2 + (g & 1)) * 512;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float a0 = (float)(int8_t)((codes >> (16 * j)) & 0xffu);
    const float a1 = (float)(int8_t)((codes >> (16 * j + 8)) & 0xffu);
    const __half2 hv = __floats2half2_rn(a0 * sc, a1 * sc);
    reinterpret_cast<uint32_t*>(frag + (gid * 4 + tig0 + j) * 16)[p] = *reinterpret_cast<const uint32_t*>(&hv);
  }
}
// act_store_corr: the accumulator seed of token t for group g, from sum = sum of its
// int8 codes over the group.
__device__ __forceinline__ void act_store_corr(uint8_t* act, int NT, int t, int g, int sum) {
  const int nt = t >> 3, tl = t & 7;
  float* cq = reinterpret_cast<float*>(act + (size_t)(g >> 1) * act_rec_bytes(NT) + NT * 1024 +
                                       ((g & 1) * NT + nt) * 64) +
              (tl >> 1) * 4 + (tl & 1);
  const float cv = (float)sum * -4.76837158203125e-07f;  // -8 * 2^-24 * sum
  cq[0] = cv;
  cq[2] = cv;
}

}  // namespace w4a8
