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
constexpr int kChunkBatch = 2;           // 64-input chunks per pipeline stage
constexpr int kPersistentCtas = 304;     // fixed constant (2 x 152 SMs): part of the canonical schedule
constexpr double kUnitFixedChunks = 3.0;  // modelled per-unit overhead, in chunk-streaming times
}  // namespace

MatmulPlan mm_plan(int K, int N) {
  MatmulPlan p;
  p.N = N;
  p.K = K;
  p.KC = chunks_of(K);
  const int n16 = N / 16;
  p.n_rg = (n16 + kGroupBlocks - 1) / kGroupBlocks;
  // Work unit = (row group, K slice).  Pick the slice count S that minimises the modelled
  // makespan on kPersistentCtas CTAs: waves * (chunks per unit + fixed per-unit cost).
  const int smax = p.KC / 2 > 1 ? (p.KC / 2 < 64 ? p.KC / 2 : 64) : 1;
  double best = 1e30;
  int bs = 1;
  for (int s = 1; s <= smax; ++s) {
    const int cps = (p.KC + s - 1) / s;
    const int S = (p.KC + cps - 1) / cps;
    const long long units = (long long)p.n_rg * S;
    const long long waves = (units + kPersistentCtas - 1) / kPersistentCtas;
    const double cost = (double)waves * ((double)cps + kUnitFixedChunks);
    if (cost < best - 1e-9) {
      best = cost;
      bs = s;
    }
  }
  p.cps = (p.KC + bs - 1) / bs;
  p.S = (p.KC + p.cps - 1) / p.cps;
  p.part_floats = p.S > 1 ? (size_t)p.S * N * 16 : 0;
  return p;
}

// d = A * B + c, m16n8k32, e4m3 inputs, fp32 accumulation.
__device__ __forceinline__ void mma_e4m3(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1, float c0, float c1, float c2, float c3) {
  asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

constexpr int kRowBlocksPerCta = kWarpsPerCta * kRowBlocksPerWarp;   // 16
static_assert(kRowBlocksPerCta == kGroupBlocks, "a CTA covers one row group of the tiled layout");
constexpr int kStageW = kRowBlocksPerCta * kChunkBatch * 512;         // weight bytes per stage
constexpr int kStageS = kRowBlocksPerCta * kChunkBatch * 64;          // scale bytes per stage
constexpr int kStageA = 2 * (2 * kChunkBatch) * 512;                  // fragment bytes (two 8-token tiles)
constexpr int kStageC = (2 * kChunkBatch) * 64;                       // correction bytes
constexpr int kStageBytes = kStageW + kStageS + kStageA + kStageC;
constexpr int kStages = 4;
constexpr int kMmThreads = 32 * (kWarpsPerCta + 1);                  // + one producer warp
constexpr size_t kMmSmem = (size_t)kStages * kStageBytes;

// Persistent CTAs: kWarpsPerCta consumer warps (kRowBlocksPerWarp 16-row blocks each) and one
// producer warp.  Work units (row group g, K slice s), unit w = g*S + s, are dealt round-robin to
// the CTAs.  The producer streams, per stage of kChunkBatch 64-input chunks, the row group's
// weights and scales, the activation fragments and the zero-point corrections into a
// kStages-deep shared-memory ring with cp.async.bulk, continuing across units; weight copies of
// the first stages are issued before griddepcontrol.wait (weights are constant), activations
// only after it.  A unit's result is folded with the other slices of its row group by the last
// unit to finish (ticket), in ascending slice order.
template <int NT>
__global__ void __launch_bounds__(kMmThreads)
    k_mm(const uint8_t* __restrict__ wt, const uint8_t* __restrict__ st, const uint8_t* __restrict__ af,
         const uint8_t* __restrict__ corr, const float* __restrict__ a_s, int M, int N, int ldy, int KC, int cps,
         int S, float* __restrict__ y, int epi, float* __restrict__ part, unsigned* __restrict__ tickets,
         unsigned* __restrict__ err, const unsigned* __restrict__ stop) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full[kStages], empty[kStages];
  __shared__ unsigned s_ticket;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n16 = N / 16;
  const int Gp = 2 * KC;  // padded groups
  const int n_rg = (n16 + kGroupBlocks - 1) / kGroupBlocks;
  const int units = n_rg * S;
  // batches of unit w (the slice's chunk range split into stages)
  auto unit_batches = [&](int w) {
    const int sl = w % S;
    const int c0 = sl * cps, c1 = min(KC, c0 + cps);
    return (c1 - c0 + kChunkBatch - 1) / kChunkBatch;
  };
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kWarpsPerCta);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  }
  __syncthreads();
  bool ok = true;

  if (warp == kWarpsPerCta) {
    // ---------------- producer ----------------
    if (lane == 0) {
      // batch sequence of this CTA: units blockIdx.x, +gridDim.x, ...; each unit's batches
      struct Pos {
        int w, b;
      };
      auto batch_info = [&](Pos ps, int& g, int& cb, int& nc, int& nrb) {
        const int sl = ps.w % S;
        g = ps.w / S;
        const int c0 = sl * cps, c1 = min(KC, c0 + cps);
        cb = c0 + ps.b * kChunkBatch;
        nc = min(kChunkBatch, c1 - cb);
        nrb = min(kGroupBlocks, n16 - g * kGroupBlocks);
      };
      auto next = [&](Pos ps) {
        if (ps.b + 1 < unit_batches(ps.w)) return Pos{ps.w, ps.b + 1};
        return Pos{ps.w + (int)gridDim.x, 0};
      };
      auto issue_weights = [&](Pos ps, int it) {
        int g, cb, nc, nrb;
        batch_info(ps, g, cb, nc, nrb);
        const int stg = it % kStages;
        mbar_expect_tx(&full[stg], (unsigned)(nrb * nc * (512 + 64) + NT * nc * 1024 + nc * 128));
        uint8_t* sw = smem + (size_t)stg * kStageBytes;
        const size_t t0 = tile_index(N, KC, g * kGroupBlocks, cb);  // contiguous stage range
        bulk_g2s(sw, wt + t0 * 512, (unsigned)(nc * nrb * 512), &full[stg]);
        bulk_g2s(sw + kStageW, st + t0 * 64, (unsigned)(nc * nrb * 64), &full[stg]);
      };
      auto issue_acts = [&](Pos ps, int it) {
        int g, cb, nc, nrb;
        batch_info(ps, g, cb, nc, nrb);
        const int stg = it % kStages;
        uint8_t* sa = smem + (size_t)stg * kStageBytes + kStageW + kStageS;
        for (int nt = 0; nt < NT; ++nt)
          bulk_g2s(sa + nt * (2 * kChunkBatch * 512), af + ((size_t)nt * Gp + 2 * cb) * 512, (unsigned)(nc * 1024),
                   &full[stg]);
        bulk_g2s(sa + kStageA, corr + (size_t)(2 * cb) * 64, (unsigned)(nc * 128), &full[stg]);
      };
      Pos pro[kStages];
      int npro = 0;
      Pos ps{(int)blockIdx.x, 0};
      while (npro < kStages && ps.w < units) {
        issue_weights(ps, npro);
        pro[npro++] = ps;
        ps = next(ps);
      }
      griddep_wait();
      int issued = npro;
      if (stop != nullptr && (__ldcg(stop) & FLAG_STOP_MASK)) {
        for (int i = 0; i < npro; ++i) issue_acts(pro[i], i);  // complete the in-flight stages, then drain
      } else {
        for (int i = 0; i < npro; ++i) issue_acts(pro[i], i);
        for (int it = npro; ps.w < units && ok; ++it) {
          const int stg = it % kStages;
          ok = mbar_wait(&empty[stg], ((it / kStages) - 1) & 1);
          if (!ok) {
            atomicOr(err, FLAG_ERR_TIMEOUT);
            break;
          }
          issue_weights(ps, it);
          issue_acts(ps, it);
          ++issued;
          ps = next(ps);
        }
      }
      // drain: every issued stage must land before the CTA may exit
      for (int it = max(0, issued - kStages); it < issued; ++it) {
        if (!mbar_wait(&full[it % kStages], (it / kStages) & 1)) {
          atomicOr(err, FLAG_ERR_TIMEOUT);
          break;
        }
      }
    }
  } else {
    // ---------------- consumers ----------------
    const int gid = lane >> 2, tig = lane & 3;
    griddep_wait();
    if (stop != nullptr && (__ldcg(stop) & FLAG_STOP_MASK)) return;
    int it = 0;  // batch counter of this CTA (ring position)
    // A failed (timed-out) wait marks the CTA broken: it then skips waits and compute but
    // keeps every barrier of the remaining units so that no warp is left waiting.
    for (int w = blockIdx.x; w < units; w += gridDim.x) {
      const int g = w / S, sl = w % S;
      const int nrb = min(kGroupBlocks, n16 - g * kGroupBlocks);
      const int c0 = sl * cps, c1 = min(KC, c0 + cps);
      const int nb = (c1 - c0 + kChunkBatch - 1) / kChunkBatch;
      const int rb0 = g * kGroupBlocks + warp * kRowBlocksPerWarp;
      float acc[kRowBlocksPerWarp][NT][4];
#pragma unroll
      for (int r = 0; r < kRowBlocksPerWarp; ++r)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[r][nt][e] = 0.0f;
      for (int b = 0; b < nb; ++b, ++it) {
        const int stg = it % kStages;
        if (ok && !mbar_wait(&full[stg], (it / kStages) & 1)) {
          if (lane == 0) atomicOr(err, FLAG_ERR_TIMEOUT);
          ok = false;
        }
        if (!ok) continue;
        const uint8_t* sw = smem + (size_t)stg * kStageBytes;
        const uint8_t* ss = sw + kStageW;
        const uint8_t* sa = ss + kStageS;
        const uint8_t* sc = sa + kStageA;
        const int nc = min(kChunkBatch, c1 - (c0 + b * kChunkBatch));
#pragma unroll
        for (int u = 0; u < kChunkBatch; ++u) {
          if (u >= nc) break;
          uint32_t av[kRowBlocksPerWarp][2][4];  // A fragments per row block and group
          float2 sg[kRowBlocksPerWarp][2];        // (row gid, row gid+8) scales per group
#pragma unroll
          for (int r = 0; r < kRowBlocksPerWarp; ++r) {
            const int rl = min(warp * kRowBlocksPerWarp + r, nrb - 1);  // idle warps read a valid tile
            const uint4 wv = reinterpret_cast<const uint4*>(sw + (u * nrb + rl) * 512)[lane];
            const uint2 sv = reinterpret_cast<const uint2*>(ss + (u * nrb + rl) * 64)[gid];
            sg[r][0] = __half22float2(*reinterpret_cast<const __half2*>(&sv.x));
            sg[r][1] = __half22float2(*reinterpret_cast<const __half2*>(&sv.y));
            // word x/z: row gid of groups 0/1; y/w: row gid+8
            av[r][0][0] = wv.x & 0x0F0F0F0Fu; av[r][0][2] = (wv.x >> 4) & 0x0F0F0F0Fu;
            av[r][0][1] = wv.y & 0x0F0F0F0Fu; av[r][0][3] = (wv.y >> 4) & 0x0F0F0F0Fu;
            av[r][1][0] = wv.z & 0x0F0F0F0Fu; av[r][1][2] = (wv.z >> 4) & 0x0F0F0F0Fu;
            av[r][1][1] = wv.w & 0x0F0F0F0Fu; av[r][1][3] = (wv.w >> 4) & 0x0F0F0F0Fu;
          }
          uint4 bf[2][NT];
          float2 cr[2][NT];
#pragma unroll
          for (int gg = 0; gg < 2; ++gg)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              bf[gg][nt] = reinterpret_cast<const uint4*>(sa + nt * (2 * kChunkBatch * 512) + (2 * u + gg) * 512)[lane];
              // negated zero-point corrections of tokens 2*tig, 2*tig+1 (see act_prep)
              cr[gg][nt] = reinterpret_cast<const float2*>(sc + (2 * u + gg) * 64)[nt * 4 + tig];
            }
          // independent MMAs first: codes x lo, starting from the correction; every partial
          // value is an integer times 2^-9 below 2^16 in magnitude, so accumulation is exact
          float d[kRowBlocksPerWarp][2][NT][4];
#pragma unroll
          for (int r = 0; r < kRowBlocksPerWarp; ++r)
#pragma unroll
            for (int gg = 0; gg < 2; ++gg)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma_e4m3(d[r][gg][nt], av[r][gg][0], av[r][gg][1], av[r][gg][2], av[r][gg][3], bf[gg][nt].z,
                         bf[gg][nt].w, cr[gg][nt].x, cr[gg][nt].y, cr[gg][nt].x, cr[gg][nt].y);
          // + codes x 16*hi
#pragma unroll
          for (int r = 0; r < kRowBlocksPerWarp; ++r)
#pragma unroll
            for (int gg = 0; gg < 2; ++gg)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma_e4m3(d[r][gg][nt], av[r][gg][0], av[r][gg][1], av[r][gg][2], av[r][gg][3], bf[gg][nt].x,
                         bf[gg][nt].y, d[r][gg][nt][0], d[r][gg][nt][1], d[r][gg][nt][2], d[r][gg][nt][3]);
          // scale and accumulate, groups in ascending order
#pragma unroll
          for (int gg = 0; gg < 2; ++gg)
#pragma unroll
            for (int r = 0; r < kRowBlocksPerWarp; ++r)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                acc[r][nt][0] = fmaf(sg[r][gg].x, d[r][gg][nt][0], acc[r][nt][0]);
                acc[r][nt][1] = fmaf(sg[r][gg].x, d[r][gg][nt][1], acc[r][nt][1]);
                acc[r][nt][2] = fmaf(sg[r][gg].y, d[r][gg][nt][2], acc[r][nt][2]);
                acc[r][nt][3] = fmaf(sg[r][gg].y, d[r][gg][nt][3], acc[r][nt][3]);
              }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stg]);
      }
      // ---- unit epilogue
      if (S > 1) {
#pragma unroll
        for (int r = 0; r < kRowBlocksPerWarp; ++r) {
          if (rb0 + r >= n16) continue;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int t0 = nt * 8 + 2 * tig;
            const int rowA = (rb0 + r) * 16 + gid;
            *reinterpret_cast<float2*>(part + ((size_t)sl * N + rowA) * 16 + t0) =
                make_float2(acc[r][nt][0], acc[r][nt][1]);
            *reinterpret_cast<float2*>(part + ((size_t)sl * N + rowA + 8) * 16 + t0) =
                make_float2(acc[r][nt][2], acc[r][nt][3]);
          }
        }
        __threadfence();
        asm volatile("bar.sync 1, %0;" ::"r"(32 * kWarpsPerCta) : "memory");
        if (threadIdx.x == 0) s_ticket = atomicAdd(tickets + g, 1u);
        asm volatile("bar.sync 1, %0;" ::"r"(32 * kWarpsPerCta) : "memory");
        if (s_ticket != (unsigned)(S - 1)) continue;  // not the last slice of this row group
        __threadfence();
#pragma unroll
        for (int r = 0; r < kRowBlocksPerWarp; ++r) {
          if (rb0 + r >= n16) continue;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int t0 = nt * 8 + 2 * tig;
            const int rowA = (rb0 + r) * 16 + gid;
            // fold slices left in ascending order; loads are issued 8 slices at a time
            float f[4];
            for (int sb = 0; sb < S; sb += 8) {
              float2 pa[8], pb[8];
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const int ss2 = sb + q;
                if (ss2 < S && ss2 != sl) {
                  pa[q] = __ldcg(reinterpret_cast<const float2*>(part + ((size_t)ss2 * N + rowA) * 16 + t0));
                  pb[q] = __ldcg(reinterpret_cast<const float2*>(part + ((size_t)ss2 * N + rowA + 8) * 16 + t0));
                } else {
                  pa[q] = make_float2(acc[r][nt][0], acc[r][nt][1]);
                  pb[q] = make_float2(acc[r][nt][2], acc[r][nt][3]);
                }
              }
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const int ss2 = sb + q;
                if (ss2 >= S) break;
                if (ss2 == 0) {
                  f[0] = pa[q].x; f[1] = pa[q].y; f[2] = pb[q].x; f[3] = pb[q].y;
                } else {
                  f[0] += pa[q].x; f[1] += pa[q].y; f[2] += pb[q].x; f[3] += pb[q].y;
                }
              }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[r][nt][e] = f[e];
          }
        }
        if (threadIdx.x == 0) tickets[g] = 0u;
      }
      if (!ok) continue;
#pragma unroll
      for (int r = 0; r < kRowBlocksPerWarp; ++r) {
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
    griddep_launch();
  }
}

cudaError_t mm_configure() {
  cudaError_t e = cudaFuncSetAttribute(k_mm<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMmSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_mm<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMmSmem);
}

cudaError_t mm_run(const MatmulPlan& p, const uint32_t* wt, const uint16_t* st, const uint4* afrag,
                   const float* corr, const float* a_s, int M, float* y, int ldy, int epi, float* part,
                   unsigned* tickets, unsigned* err, const unsigned* stop, cudaStream_t stream) {
  static cudaError_t configured = mm_configure();
  if (configured != cudaSuccess) return configured;
  const long long units = (long long)p.n_rg * p.S;
  dim3 grid((unsigned)(units < kPersistentCtas ? units : kPersistentCtas));
  dim3 block(kMmThreads);
  const uint8_t* w8 = reinterpret_cast<const uint8_t*>(wt);
  const uint8_t* s8 = reinterpret_cast<const uint8_t*>(st);
  const uint8_t* a8 = reinterpret_cast<const uint8_t*>(afrag);
  const uint8_t* c8 = reinterpret_cast<const uint8_t*>(corr);
  if (M <= 8)
    return launch_pdl(k_mm<1>, grid, block, kMmSmem, stream, w8, s8, a8, c8, a_s, M, p.N, ldy, p.KC, p.cps, p.S, y,
                      epi, part, tickets, err, stop);
  return launch_pdl(k_mm<2>, grid, block, kMmSmem, stream, w8, s8, a8, c8, a_s, M, p.N, ldy, p.KC, p.cps, p.S, y,
                    epi, part, tickets, err, stop);
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
    af[((size_t)nt * Gp + g) * 32 + lane] = make_uint4(hi0, hi1, lo0, lo1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    if (tig == 0) corr[(size_t)g * 16 + t] = (float)sum * -0.015625f;  // -8 * sum * 2^-9
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
  size_t off_afrag, off_corr, off_part, off_tickets, off_err, total;
};
inline size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }
MatmulWorkspace ws_layout(const MatmulPlan& p) {
  MatmulWorkspace w;
  w.off_afrag = 0;
  w.off_corr = align256(w.off_afrag + afrag_uint4(p.K) * 16);
  w.off_part = align256(w.off_corr + corr_floats(p.K) * 4);
  w.off_tickets = align256(w.off_part + p.part_floats * 4);
  w.off_err = align256(w.off_tickets + (size_t)p.n_rg * 4);
  w.total = w.off_err + 256;
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
  if (!aligned(w_t, 16) || !aligned(s_t, 16) || !aligned(workspace, 256) || !aligned(a_q, 4)) return W4A8_ERR_ARG;
  const MatmulPlan p = mm_plan(K, N);
  const MatmulWorkspace w = ws_layout(p);
  if (workspace_bytes < w.total) return W4A8_ERR_CAPACITY;
  if (!aligned(a_s, 4)) return W4A8_ERR_ARG;
  char* base = static_cast<char*>(workspace);
  uint4* af = reinterpret_cast<uint4*>(base + w.off_afrag);
  float* corr = reinterpret_cast<float*>(base + w.off_corr);
  float* part = reinterpret_cast<float*>(base + w.off_part);
  unsigned* tickets = reinterpret_cast<unsigned*>(base + w.off_tickets);
  unsigned* err = reinterpret_cast<unsigned*>(base + w.off_err);
  cudaStream_t st = as_stream(stream);
  W4A8_CUDA_TRY(act_prep_run(a_q, M, K, K, af, corr, tickets, p.n_rg, st));
  W4A8_CUDA_TRY(mm_run(p, w_t, s_t, af, corr, a_s, M, y, N, EPI_STORE, part, tickets, err, nullptr, st));
  return W4A8_OK;
}

W4A8_API w4a8_status w4a8_matmul_check(const void* workspace, int M, int K, int N, uint32_t* flags) {
  if (!workspace || !flags || M <= 0 || K <= 0 || N <= 0) return W4A8_ERR_ARG;
  if (M > 16 || K % 32 || N % 16) return W4A8_ERR_SHAPE;
  const MatmulWorkspace w = ws_layout(mm_plan(K, N));
  const char* base = static_cast<const char*>(workspace);
  W4A8_CUDA_TRY(cudaMemcpy(flags, base + w.off_err, 4, cudaMemcpyDeviceToHost));
  return *flags ? W4A8_ERR_DEVICE_FLAG : W4A8_OK;
}
