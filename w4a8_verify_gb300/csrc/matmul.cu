// W4A8 small-batch matmul on the legacy tensor-core path (mma.sync m16n8k32 e4m3).
//
// "GPU-Resident Speculative Decoding ..." (Design > Small-Batch Verification Kernels):
// verification multiplies every weight matrix by a handful of token vectors, so it
// reads the same weight bytes as a single-token step; one weight load serves every
// token; the zero point of the 4-bit codes is removed with a per-block correction
// term.  Implementation (deterministic mode): the reduction order is fixed for every
// token count, so N tokens give the bits of N single-token steps.
//
// GB300 design: the integer dot products run on the tensor cores instead of dp4a.
// Weight codes n = q + 8 enter as e4m3 bytes n * 2^-9 (one AND per four codes), an int8
// activation a enters as the exact pair (16*hi, lo) of e4m3 values, so every MMA
// partial sum is an exact integer times 2^-9 and the group sum
//   isum = 2^9 * (mma(n, 16hi) + mma(n, lo)) - 8 * sum(a)
// is exact.  Each group's isum is scaled by its fp16 weight scale with one fmaf in a
// fixed order; the schedule (slices of K) depends on (K, N) only.
#include "matmul.cuh"

namespace w4a8 {

namespace {
constexpr int kChunkBatch = 4;  // 64-input chunks loaded per warp before computing
constexpr int kTargetCtas = 608;  // fixed constant (4 x 152): part of the canonical schedule
}  // namespace

MatmulPlan mm_plan(int K, int N) {
  MatmulPlan p;
  p.N = N;
  p.K = K;
  p.KC = chunks_of(K);
  const int n16 = N / 16;
  p.n_rg = (n16 + kWarpsPerCta * kRowBlocksPerWarp - 1) / (kWarpsPerCta * kRowBlocksPerWarp);
  int s = (kTargetCtas + p.n_rg / 2) / p.n_rg;
  int smax = p.KC / 2 > 1 ? p.KC / 2 : 1;  // at least two chunks per slice
  if (s < 1) s = 1;
  if (s > smax) s = smax;
  p.cps = (p.KC + s - 1) / s;
  p.S = (p.KC + p.cps - 1) / p.cps;
  p.part_floats = p.S > 1 ? (size_t)p.S * N * 16 : 0;
  return p;
}

__device__ __forceinline__ void mma_e4m3(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int NT, int R>
__global__ void __launch_bounds__(32 * kWarpsPerCta)
    k_mm(const uint4* __restrict__ wt, const uint2* __restrict__ st, const uint4* __restrict__ af,
         const float* __restrict__ corr, const float* __restrict__ a_s, int M, int N, int ldy, int KC, int cps,
         int S, float* __restrict__ y, int epi, float* __restrict__ part, unsigned* __restrict__ tickets) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int n16 = N / 16;
  const int rb0 = (blockIdx.x * kWarpsPerCta + warp) * R;
  const int s = blockIdx.y;
  const int c0 = s * cps;
  const int c1 = min(KC, c0 + cps);

  float acc[R][NT][4];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[r][nt][e] = 0.0f;

  bool waited = false;
  for (int cb = c0; cb < c1; cb += kChunkBatch) {
    uint4 wv[kChunkBatch][R];
    uint2 sv[kChunkBatch][R];
#pragma unroll
    for (int u = 0; u < kChunkBatch; ++u)
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int c = cb + u;
        if (c < c1 && rb0 + r < n16) {
          const size_t base = (size_t)(rb0 + r) * KC + c;
          wv[u][r] = __ldg(wt + base * 32 + lane);
          sv[u][r] = __ldg(st + base * 8 + gid);
        } else {
          wv[u][r] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
          sv[u][r] = make_uint2(0u, 0u);
        }
      }
    if (!waited) {  // weights are constant: their first loads overlap the previous kernel
      griddep_wait();
      waited = true;
    }
#pragma unroll
    for (int u = 0; u < kChunkBatch; ++u) {
      const int c = cb + u;
      if (c >= c1) break;
#pragma unroll
      for (int gg = 0; gg < 2; ++gg) {
        const int g = 2 * c + gg;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint4 b = __ldg(af + ((size_t)g * 2 + nt) * 32 + lane);
          const float2 cr = __ldg(reinterpret_cast<const float2*>(corr + (size_t)g * 16 + nt * 8 + 2 * tig));
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const uint32_t wA = gg ? wv[u][r].z : wv[u][r].x;  // row gid
            const uint32_t wB = gg ? wv[u][r].w : wv[u][r].y;  // row gid + 8
            const uint32_t a0 = wA & 0x0F0F0F0Fu, a2 = (wA >> 4) & 0x0F0F0F0Fu;
            const uint32_t a1 = wB & 0x0F0F0F0Fu, a3 = (wB >> 4) & 0x0F0F0F0Fu;
            float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            mma_e4m3(d, a0, a1, a2, a3, b.x, b.y);  // codes x 16*hi
            mma_e4m3(d, a0, a1, a2, a3, b.z, b.w);  // codes x lo
            const uint32_t sp = gg ? sv[u][r].y : sv[u][r].x;
            const float sA = __half2float(__ushort_as_half((unsigned short)(sp & 0xffffu)));
            const float sB = __half2float(__ushort_as_half((unsigned short)(sp >> 16)));
            acc[r][nt][0] = fmaf(sA, d[0] - cr.x, acc[r][nt][0]);
            acc[r][nt][1] = fmaf(sA, d[1] - cr.y, acc[r][nt][1]);
            acc[r][nt][2] = fmaf(sB, d[2] - cr.x, acc[r][nt][2]);
            acc[r][nt][3] = fmaf(sB, d[3] - cr.y, acc[r][nt][3]);
          }
        }
      }
    }
  }
  if (!waited) griddep_wait();
  griddep_launch();

  bool finalize = true;
  if (S > 1) {
    // write this slice's partial, then the last CTA of the row group folds all slices
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (rb0 + r >= n16) continue;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int t0 = nt * 8 + 2 * tig;
        const int rowA = (rb0 + r) * 16 + gid;
        float* pa = part + ((size_t)s * N + rowA) * 16 + t0;
        float* pb = part + ((size_t)s * N + rowA + 8) * 16 + t0;
        *reinterpret_cast<float2*>(pa) = make_float2(acc[r][nt][0], acc[r][nt][1]);
        *reinterpret_cast<float2*>(pb) = make_float2(acc[r][nt][2], acc[r][nt][3]);
      }
    }
    __threadfence();
    __syncthreads();
    __shared__ unsigned s_ticket;
    if (threadIdx.x == 0) s_ticket = atomicAdd(tickets + blockIdx.x, 1u);
    __syncthreads();
    finalize = (s_ticket == (unsigned)(S - 1));
    if (finalize) {
      __threadfence();
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (rb0 + r >= n16) continue;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int t0 = nt * 8 + 2 * tig;
          const int rowA = (rb0 + r) * 16 + gid;
          float f[4];
#pragma unroll
          for (int ss = 0; ss < S; ++ss) {
            float2 pa, pb;
            if (ss == s) {
              pa = make_float2(acc[r][nt][0], acc[r][nt][1]);
              pb = make_float2(acc[r][nt][2], acc[r][nt][3]);
            } else {
              pa = __ldcg(reinterpret_cast<const float2*>(part + ((size_t)ss * N + rowA) * 16 + t0));
              pb = __ldcg(reinterpret_cast<const float2*>(part + ((size_t)ss * N + rowA + 8) * 16 + t0));
            }
            if (ss == 0) {
              f[0] = pa.x; f[1] = pa.y; f[2] = pb.x; f[3] = pb.y;
            } else {
              f[0] += pa.x; f[1] += pa.y; f[2] += pb.x; f[3] += pb.y;
            }
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[r][nt][e] = f[e];
        }
      }
      if (threadIdx.x == 0) tickets[blockIdx.x] = 0u;
    }
  }
  if (!finalize) return;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (rb0 + r >= n16) continue;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = nt * 8 + 2 * tig + (e & 1);
        if (t >= M) continue;
        const int row = (rb0 + r) * 16 + gid + ((e & 2) ? 8 : 0);
        const float v = acc[r][nt][e] * (512.0f * __ldg(a_s + t));
        float* dst = y + (size_t)t * ldy + row;
        if (epi == EPI_ADD)
          *dst = *dst + v;
        else
          *dst = v;
      }
    }
  }
}

cudaError_t mm_run(const MatmulPlan& p, const uint32_t* wt, const uint16_t* st, const uint4* afrag,
                   const float* corr, const float* a_s, int M, float* y, int ldy, int epi, float* part,
                   unsigned* tickets, cudaStream_t stream) {
  dim3 grid(p.n_rg, p.S);
  dim3 block(32 * kWarpsPerCta);
  const uint4* w4 = reinterpret_cast<const uint4*>(wt);
  const uint2* s2 = reinterpret_cast<const uint2*>(st);
  if (M <= 8)
    return launch_pdl(k_mm<1, kRowBlocksPerWarp>, grid, block, 0, stream, w4, s2, afrag, corr, a_s, M, p.N, ldy,
                      p.KC, p.cps, p.S, y, epi, part, tickets);
  return launch_pdl(k_mm<2, kRowBlocksPerWarp>, grid, block, 0, stream, w4, s2, afrag, corr, a_s, M, p.N, ldy,
                    p.KC, p.cps, p.S, y, epi, part, tickets);
}

// One warp per padded group: fragment bytes and zero-point corrections of 16 tokens.
__global__ void k_act_prep(const int8_t* __restrict__ a_q, int M, int K, int lda, uint4* __restrict__ af,
                           float* __restrict__ corr, unsigned* __restrict__ tickets, int n_tickets) {
  griddep_wait();
  const int gtid = blockIdx.x * blockDim.x + threadIdx.x;
  for (int i = gtid; i < n_tickets; i += gridDim.x * blockDim.x) tickets[i] = 0u;
  const int Gp = groups_padded(K), G = K / 32;
  const int g = gtid >> 5;
  if (g >= Gp) return;
  const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int t = nt * 8 + gid;
    uint32_t hi0 = 0, hi1 = 0, lo0 = 0, lo1 = 0;
    int sum = 0;
    if (t < M && g < G) {
      const int8_t* src = a_q + (size_t)t * lda + 32 * g + 4 * tig;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        uint32_t hb, lb;
        const int a0 = src[b];
        split_act(a0, hb, lb);
        hi0 |= hb << (8 * b);
        lo0 |= lb << (8 * b);
        const int a1 = src[16 + b];
        split_act(a1, hb, lb);
        hi1 |= hb << (8 * b);
        lo1 |= lb << (8 * b);
        sum += a0 + a1;
      }
    }
    af[((size_t)g * 2 + nt) * 32 + lane] = make_uint4(hi0, hi1, lo0, lo1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    if (tig == 0) corr[(size_t)g * 16 + t] = (float)sum * 0.015625f;  // 8 * sum * 2^-9
  }
}

cudaError_t act_prep_run(const int8_t* a_q, int M, int K, int lda, uint4* afrag, float* corr, unsigned* tickets,
                         int n_tickets, cudaStream_t stream) {
  const int Gp = groups_padded(K);
  const int threads = 128;
  const int blocks = (Gp * 32 + threads - 1) / threads;
  return launch_pdl(k_act_prep, dim3(blocks), dim3(threads), 0, stream, a_q, M, K, lda, afrag, corr, tickets,
                    n_tickets);
}

}  // namespace w4a8

using namespace w4a8;

namespace {
struct MatmulWorkspace {
  size_t off_afrag, off_corr, off_part, off_tickets, total;
};
inline size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }
MatmulWorkspace ws_layout(const MatmulPlan& p) {
  MatmulWorkspace w;
  w.off_afrag = 0;
  w.off_corr = align256(w.off_afrag + afrag_uint4(p.K) * 16);
  w.off_part = align256(w.off_corr + corr_floats(p.K) * 4);
  w.off_tickets = align256(w.off_part + p.part_floats * 4);
  w.total = align256(w.off_tickets + (size_t)p.n_rg * 4);
  return w;
}
}  // namespace

W4A8_API int w4a8_matmul_slices(int K, int N) {
  if (K <= 0 || N <= 0 || K % 32 || N % 16) return 0;
  return mm_plan(K, N).S;
}

W4A8_API w4a8_status w4a8_matmul_workspace_bytes(int M, int K, int N, size_t* bytes) {
  if (!bytes || M <= 0 || K <= 0 || N <= 0) return W4A8_ERR_ARG;
  if (M > 16 || K % 32 || N % 16) return W4A8_ERR_SHAPE;
  *bytes = ws_layout(mm_plan(K, N)).total;
  return W4A8_OK;
}

W4A8_API w4a8_status w4a8_matmul(const int8_t* a_q, const float* a_s, int M, int K, const uint32_t* w_t,
                                 const uint16_t* s_t, int N, float* y, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  if (!a_q || !a_s || !w_t || !s_t || !y || !workspace || M <= 0 || K <= 0 || N <= 0) return W4A8_ERR_ARG;
  if (M > 16 || K % 32 || N % 16) return W4A8_ERR_SHAPE;
  if (!aligned(w_t, 16) || !aligned(s_t, 8) || !aligned(workspace, 256) || !aligned(a_q, 4)) return W4A8_ERR_ARG;
  const MatmulPlan p = mm_plan(K, N);
  const MatmulWorkspace w = ws_layout(p);
  if (workspace_bytes < w.total) return W4A8_ERR_CAPACITY;
  char* base = static_cast<char*>(workspace);
  uint4* af = reinterpret_cast<uint4*>(base + w.off_afrag);
  float* corr = reinterpret_cast<float*>(base + w.off_corr);
  float* part = reinterpret_cast<float*>(base + w.off_part);
  unsigned* tickets = reinterpret_cast<unsigned*>(base + w.off_tickets);
  cudaStream_t st = as_stream(stream);
  W4A8_CUDA_TRY(act_prep_run(a_q, M, K, K, af, corr, tickets, p.n_rg, st));
  W4A8_CUDA_TRY(mm_run(p, w_t, s_t, af, corr, a_s, M, y, N, EPI_STORE, part, tickets, st));
  return W4A8_OK;
}
