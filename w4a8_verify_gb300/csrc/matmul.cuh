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

// Output handling after the fixed-order reduction: y = fold * s_a[t], then
enum MatmulEpilogue : int {
  EPI_STORE = 0,  // y[t][n] = value
  EPI_ADD = 1,    // y[t][n] += value (residual stream)
};

// Launches the matmul kernel on prepared activation fragments.  part/tickets: split-K
// scratch (part_floats floats, n_rg counters that must be zero on entry; the kernel
// leaves them zero).
// Raises the dynamic shared-memory limit of the matmul kernels (call once per device,
// outside stream capture).
cudaError_t mm_configure();

// err: device word that receives FLAG_ERR_TIMEOUT if a bounded pipeline wait expires.
// stop: optional device control word; when it has a FLAG_STOP_MASK bit set at kernel
// start (after the dependency wait) the kernel does nothing.
cudaError_t mm_run(const MatmulPlan& p, const uint32_t* wt, const uint16_t* st, const uint4* afrag,
                   const float* corr, const float* a_s, int M, float* y, int ldy, int epi, float* part,
                   unsigned* tickets, unsigned* err, const unsigned* stop, cudaStream_t stream);

// P2 layout (rows [0, N)) -> rows [row0, row0 + N) of an Ntot-row tiled matrix (quant.cu).
cudaError_t repack_run(const uint32_t* w_p2, const uint16_t* s_p2, int N, int K, int Ntot, int row0, uint32_t* w_t,
                       uint16_t* s_t, cudaStream_t st);

// Launches the fragment builder for int8 activations a_q[M][K] (row stride lda) and zeroes
// n_tickets counters.
cudaError_t act_prep_run(const int8_t* a_q, int M, int K, int lda, uint4* afrag, float* corr,
                         unsigned* tickets, int n_tickets, cudaStream_t stream);

// Device helper for fused producers: writes the fragment bytes of one 4-input quad.
// For token t (< 16) and inputs k0..k0+3 (k0 % 4 == 0) with int8 codes in `codes`
// (byte b = input k0+b), stores the hi and lo e4m3 bytes into the fragment buffer of an
// input dimension with Gp padded groups (layout [8-token tile][Gp][32 lanes] uint4).
__device__ __forceinline__ void afrag_store_quad(uint4* afrag, int Gp, int t, int k0, uint32_t codes) {
  const int g = k0 >> 5;
  const int kin = k0 & 31;              // 0..28
  const int tig = (kin & 15) >> 2;
  const int upper = kin >> 4;           // 0: inputs 4tig..4tig+3, 1: inputs 16+4tig..
  const int nt = t >> 3, gid = t & 7;
  uint32_t hi = 0, lo = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const int a = (int)(int8_t)((codes >> (8 * b)) & 0xffu);
    uint32_t hb, lb;
    split_act(a, hb, lb);
    hi |= hb << (8 * b);
    lo |= lb << (8 * b);
  }
  uint32_t* dst = reinterpret_cast<uint32_t*>(afrag + ((size_t)nt * Gp + g) * 32 + gid * 4 + tig);
  dst[upper] = hi;
  dst[2 + upper] = lo;
}

}  // namespace w4a8
