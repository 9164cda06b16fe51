// Tree attention: the chunk kernel k_attn<D, G, QT, MERGE> and its launch templates, shared by
// the translation units that instantiate it (attention_d64.cu, attention_d128.cu) and by
// layers.cu (host entry points, the merge kernel).
//
// "GPU-Resident Speculative Decoding ..." (Design > GPU-Resident Speculation Loop): each tree
// node attends to the committed cache and to its ancestors; (Design > Small-Batch
// Verification Kernels): the visible context is split into chunks that separate CTAs process
// and a second pass merges; the query heads that share a KV head read each key and value once.
#pragma once
#include "decoder.cuh"
#include "layers.cuh"

namespace w4a8 {

__device__ __forceinline__ bool stopped(const SpecCtl* ctl) { return (ctl->flags & FLAG_STOP_MASK) != 0u; }

// ---------------------------------------------------------------------- tree attention

constexpr int kAttnStages = 2;                      // chunks in flight (K and V entries of 64 rows each)
constexpr int kAttnWarps = 8;                       // compute warps; one more warp issues the copies
constexpr int kAttnThreads = 32 * (kAttnWarps + 1);
constexpr float kAttnEScale = 32768.0f;             // 2^15: weights e in [0, 1] enter the value product scaled
// Shared-memory row strides (floats) of a ring entry: key rows D + 8 and value rows D + 4, so
// that the B fragments (rows 2t.., columns g) of the tensor-core steps fall on distinct banks;
// score rows kAttnChunk + 8, so that the float2 score stores of a fragment do as well.
__host__ __device__ constexpr int attn_kstr(int D) { return D + 8; }
__host__ __device__ constexpr int attn_vstr(int D) { return D + 4; }
constexpr int kAttnSpStr = kAttnChunk + 8;

// Shared-memory carve-up of the chunk kernel for head size D and at most QN queries.
struct AttnLayout {
  size_t stage, q, kt, vt, sp, ef, total;
};
__host__ __device__ inline AttnLayout attn_layout(int D, int QN) {
  AttnLayout a;
  const size_t nmt = (size_t)(QN + 15) / 16;
  a.stage = (size_t)kAttnChunk * (attn_kstr(D) + attn_vstr(D)) * 4;  // ring entry 2s: K rows, 2s + 1: V rows
  a.q = kAttnStages * a.stage;                       // query A fragments [m-tile][k-step][lane] (hi, lo)
  a.kt = a.q + nmt * (D / 16) * 32 * 32;             // tree K rows [16][D]
  a.vt = a.kt + (size_t)kMaxWidth * D * 4;           // tree V rows
  a.sp = a.vt + (size_t)kMaxWidth * D * 4;           // scores [q][kAttnSpStr]
  a.ef = a.sp + (size_t)QN * kAttnSpStr * 4;         // weights e as A fragments [m-tile][slot step][lane] (hi, lo)
  a.total = a.ef + nmt * (kAttnChunk / 16) * 32 * 32;
  return a;
}

// Consumer-warp barrier with an AND vote (the copy warp does not take part).
__device__ __forceinline__ bool consumers_all(bool v) {
  unsigned r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((unsigned)v), "r"(32 * kAttnWarps)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(32 * kAttnWarps) : "memory");
}

// f16 pair split of two floats: hi = rn(x), lo = rn(x - hi) (x - hi is exact in f32).
__device__ __forceinline__ void split_h2(float x, float y, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x, y);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(x - hf.x, y - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}
// d = A * B + d, m16n8k16, f16 inputs, f32 accumulation.
__device__ __forceinline__ void mma_acc(float (&d)[4], uint4 a, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}
// Score contribution of one 16-dimension step: three products of the f16 splits (hi*hi,
// hi*lo, lo*hi, in this order) into the f32 accumulator.
__device__ __forceinline__ void mma_split3(float (&d)[4], uint4 ahi, uint4 alo, uint32_t bh0, uint32_t bh1,
                                           uint32_t bl0, uint32_t bl1) {
  mma_acc(d, ahi, bh0, bh1);
  mma_acc(d, ahi, bl0, bl1);
  mma_acc(d, alo, bh0, bh1);
}


// Attention pass, grid (split sp, KV head kh).  Chunks of kAttnChunk logical positions are
// dealt to the splits in contiguous ranges of R (R and the split count depend on the cache
// capacity and the head count only).  A copy warp brings each chunk's cached K and V rows
// into a ring of 2 * kAttnStages entries with one TMA box each (rows at padded strides); the
// compute warps keep, for every query of the KV head (node i, head g; q = i*G + g), a running
// (M, L, O) over its chunks in ascending order:
//   scores: s = q . k on the tensor cores (mma m16n8k16, f32 accumulation) from the f16 splits
//           q = qh + ql, k = kh + kl: per 16-dimension step qh.kh + qh.kl + ql.kh, steps in order
//           (the row of a score depends on its own query and key only);
//   per chunk: m = max(M, max over visible slots), c = exp(M - m), e_j = exp(s_j - m),
//           L = L * c + (butterfly sum of e over the 64 slots, lane l holding slots 2l, 2l+1);
//   values: O = O * c, then O += e . v on the tensor cores from the f16 splits of 2^15 e and
//           of v (per 16-slot step eh.vh + eh.vl + el.vh, steps in order; the exact factor
//           2^15 is removed when the partial is stored); M = m.
// Slots below the committed length L read the cache; slots at L + e read the node's
// ancestor at depth e (tree rows).  A 16-key or 16-slot group reaching past the cache is
// multiplied with each node's own rows (zero rows past the node), keeping that node's rows
// of the result; when every tree slot holds one row for all the nodes that see it, that row
// serves every query (a key a query does not see is masked, a value has weight zero).  Either
// way every row sees the same operations as in a step where those slots are cached.
// The last CTA of a KV head to finish (ticket) merges the splits of every query in ascending
// order (M = max M_s, L = sum exp(M_s - M) L_s, O = sum exp(M_s - M) O_s), writes O / L and
// the per-(node, head) maximum |O / L| that the quantiser of the O projection reads (MERGE;
// otherwise k_attn_merge does the same merge with one CTA per (node, head)).  Every order is
// a function of the logical position.
// (one CTA per SM: 168 registers keep the three warps of a sub-partition within its 16384)
template <int D, int G, int QT, bool MERGE>
__global__ void __maxnreg__(168)
    k_attn(SpecCtl* ctl, const TreeState* __restrict__ tree, int N, const float* __restrict__ qrot,
           const float* __restrict__ kc, const float* __restrict__ vc, int kv_cap, int Hq, int R,
           float* __restrict__ o_part, float2* __restrict__ ml_part, unsigned* __restrict__ tickets,
           float* __restrict__ out, float2* __restrict__ mpart, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_v, int layer) {
  constexpr int CH = kAttnChunk;
  constexpr int DL = D / 32;         // dimensions per lane in the merge
  constexpr int KS = D / 16;         // 16-dimension steps of a score
  constexpr int VS = CH / 16;        // 16-slot steps of the value product
  constexpr int NTW = D / 8 / kAttnWarps;  // 8-dimension n-tiles of the value product per warp
  constexpr int MT = (kMaxWidth * G + 15) / 16 < (QT + 1) / 2 ? (kMaxWidth * G + 15) / 16 : (QT + 1) / 2;
  constexpr int NE = 2 * kAttnStages;  // ring entries (K or V rows of one chunk)
  constexpr int MSPAN = (16 % G == 0) ? 1 : 2;  // m-tiles that hold one node's rows, at most
  constexpr int KSTR = attn_kstr(D), VSTR = attn_vstr(D), SPS = kAttnSpStr;
  // scores of a fully cached chunk: WPM warps per m-tile, NTPW key n-tiles (8 keys) per warp
  constexpr int WPM = kAttnWarps / MT, NTPW = (CH / 8) / WPM;
  static_assert(CH / 8 == kAttnWarps, "one key n-tile per warp in chunks reaching past the cache");
  static_assert((WPM & (WPM - 1)) == 0 && WPM * NTPW == CH / 8, "score partition");
  static_assert(D == 64 || D == 128, "head size");
  static_assert(NTW >= 1 && NTW * 8 * kAttnWarps == D, "value n-tiles");
  // The committed length, the tree shape and the cached rows below it were written by
  // earlier steps, so the copies of the cached rows start before the dependency wait (the
  // kernel just before this one writes only the tree slots and the queries).
  griddep_launch();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_path[kMaxWidth][kMaxWidth];
  __shared__ int s_dep[kMaxWidth], s_par[kMaxWidth];
  __shared__ int s_row[kMaxWidth];  // tree row at depth e shared by every node that deep, or -1
  __shared__ float s_cs[kMaxWidth * 8];  // per-query rescale c of the running values (this chunk)
  __shared__ float s_M[kMaxWidth * 8], s_L[kMaxWidth * 8];  // running max and sum per query
  __shared__ uint64_t full[NE], empty[NE];
  __shared__ unsigned s_last;
  const int kh = blockIdx.y;
  // blockIdx.z: 16-node sub-chain of a prefill bucket (0 in verification).  Sub-chain j is the
  // chain of the bucket's tokens 16j .. 16j+15: its committed length is 16j further, and its
  // queries, outputs and partials are the next 16 rows of each buffer.  Only the variants that
  // leave the merge to k_attn_merge take prefill buckets (16-node chains with G >= 2).
  const int sub = MERGE ? 0 : (int)blockIdx.z;
  if (sub > 0) {
    const size_t rows = (size_t)sub * kMaxWidth;
    qrot += rows * Hq * D;
    out += rows * Hq * D;
    mpart += rows * Hq;
    o_part += rows * gridDim.x * Hq * D;
    ml_part += rows * gridDim.x * Hq;
    tickets += (size_t)sub * gridDim.y;
  }
  const int L = (int)ctl->committed_len + sub * kMaxWidth;
  int maxd = 0;
  for (int i = 0; i < N; ++i) maxd = max(maxd, tree->depth[i]);
  const int nch = (L + maxd) / CH + 1;
  const int c_begin = blockIdx.x * R, c_end = min(nch, c_begin + R);
  if (c_begin >= nch) return;  // uniform over the CTA
  const int nsa = (nch + R - 1) / R;  // CTAs of this head that hold chunks
  const int QN = N * G;
  const int nmt = (QN + 15) / 16;
  const AttnLayout lay = attn_layout(D, QN);
  uint8_t* Qf = smem + lay.q;
  float* Kt = reinterpret_cast<float*>(smem + lay.kt);
  float* Vt = reinterpret_cast<float*>(smem + lay.vt);
  float* SP = reinterpret_cast<float*>(smem + lay.sp);
  uint32_t* EF = reinterpret_cast<uint32_t*>(smem + lay.ef);
  const float* kb = kc + (size_t)kh * kv_cap * D;
  const float* vb = vc + (size_t)kh * kv_cap * D;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lg = lane >> 2, lt = lane & 3;  // fragment row group and thread-in-group
  // ring entry e: K rows of stage e / 2 (even e) or its V rows (odd e)
  auto ring_entry = [&](int e) -> uint8_t* {
    return smem + (size_t)(e >> 1) * lay.stage + ((e & 1) ? (size_t)CH * KSTR * 4 : 0);
  };
  if (threadIdx.x == 0) {
    for (int i = 0; i < NE; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  }
  __syncthreads();

  if (warp == kAttnWarps) {
    // ---------------- copy warp: entries K(c0) V(c0) K(c1) V(c1) ..., one TMA box of 64 rows
    // each (rows land at the padded strides; columns past D and rows past the cache read zero;
    // rows between L and the chunk end are never read from the ring)
    if (lane == 0) {
      // a later sub-chain's cached rows include the rows the kernel just before this one wrote
      // for the earlier sub-chains of the bucket: wait for it before the first copy
      if (sub > 0) griddep_wait();
      int n = 0;  // entries issued
      for (int c = c_begin; c < c_end; ++c) {
        const int P0 = c * CH;
        const bool any = L > P0;  // the chunk holds cached rows
        for (int kv = 0; kv < 2; ++kv, ++n) {
          const int e = n % NE;
          if (n >= NE && !mbar_wait(&empty[e], ((n / NE) - 1) & 1)) {
            atomicOr(&ctl->flags, FLAG_ERR_TIMEOUT);
            c = c_end;
            break;
          }
          mbar_expect_tx(&full[e], any ? (unsigned)(CH * (kv ? VSTR : KSTR) * 4) : 0u);
          if (any) tma_load_4d(ring_entry(e), kv ? &tm_v : &tm_k, 0, P0, kh, layer, &full[e]);
        }
      }
      // every issued copy lands before the CTA exits
      for (int j = max(0, n - NE); j < n; ++j)
        if (!mbar_wait(&full[j % NE], (j / NE) & 1)) {
          atomicOr(&ctl->flags, FLAG_ERR_TIMEOUT);
          break;
        }
    }
    return;
  }

  // ---------------- compute warps ----------------
  // Set-up that needs only earlier steps' state (the tree shape) or nothing, before the
  // dependency wait: node depths and root paths, zeroed weight fragments (rows past QN stay
  // zero: their products are discarded), the running max and sum.
  if (threadIdx.x < N) {
    s_dep[threadIdx.x] = tree->depth[threadIdx.x];
    s_par[threadIdx.x] = tree->parent[threadIdx.x];
  }
  for (int idx = threadIdx.x; idx < nmt * VS * 32 * 8; idx += 32 * kAttnWarps) EF[idx] = 0u;
  for (int q = threadIdx.x; q < QN; q += 32 * kAttnWarps) {
    s_M[q] = -INFINITY;
    s_L[q] = 0.0f;
  }
  consumers_sync();
  if (threadIdx.x < N) {
    const int i = threadIdx.x;
    int cur = i;
    for (int e = s_dep[i]; e >= 0; --e) {
      s_path[i][e] = cur;
      cur = e > 0 ? s_par[cur] : 0;
    }
  }
  griddep_wait();
  if (!consumers_all(!stopped(ctl))) {
    // keep the ring consistent for the copy warp: consume every entry it issues
    // (error state: nothing is computed)
    int n = 0;
    for (int c = c_begin; c < c_end; ++c)
      for (int kv = 0; kv < 2; ++kv, ++n) {
        const int e = n % NE;
        const bool got = consumers_all(mbar_wait(&full[e], (n / NE) & 1));
        if (threadIdx.x == 0) mbar_arrive(&empty[e]);
        if (!got) return;
      }
    return;
  }
  // slot L + e of every node that deep holds the same row (a chain, or a shared prefix)?
  if (threadIdx.x <= maxd) {
    const int e = threadIdx.x;
    int r = -1;
    bool same = true;
    for (int i = 0; i < N; ++i)
      if (s_dep[i] >= e) {
        if (r < 0) r = s_path[i][e];
        else same = same && s_path[i][e] == r;
      }
    s_row[e] = same ? r : -1;
  }
  // queries of the KV head (the G heads of kh are consecutive in qrot) and the tree rows
  // (slots L .. L+N-1, read by the chunks that reach past L), both written by the kernel
  // just before this one; every load is issued before the first split.
  // A fragments of m16n8k16 (rows = queries, columns = dimensions), split into f16 hi and lo:
  // lane (g, t) of m-tile mt, step s holds rows g, g+8 and columns 2t, 2t+1, 2t+8, 2t+9
  {
    constexpr int QI = (MT * KS * 32 + 32 * kAttnWarps - 1) / (32 * kAttnWarps);
    float v[QI][8];
#pragma unroll
    for (int it = 0; it < QI; ++it) {
      const int idx = threadIdx.x + it * 32 * kAttnWarps;
      const int ln = idx & 31, st = (idx >> 5) % KS, mt = (idx >> 5) / KS;
      const int g = ln >> 2, t = ln & 3;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int q = mt * 16 + g + 8 * h;
        float2 lo2 = make_float2(0.0f, 0.0f), hi2 = make_float2(0.0f, 0.0f);
        if (idx < nmt * KS * 32 && q < QN) {
          const float* qr = qrot + ((size_t)(q / G) * Hq + kh * G + q % G) * D + st * 16 + 2 * t;
          lo2 = *reinterpret_cast<const float2*>(qr);
          hi2 = *reinterpret_cast<const float2*>(qr + 8);
        }
        v[it][2 * h] = lo2.x; v[it][2 * h + 1] = lo2.y; v[it][4 + 2 * h] = hi2.x; v[it][5 + 2 * h] = hi2.y;
      }
    }
    constexpr int TI = (kMaxWidth * D / 4 + 32 * kAttnWarps - 1) / (32 * kAttnWarps);
    float4 kt[TI], vt[TI];
#pragma unroll
    for (int it = 0; it < TI; ++it) {
      const int idx = threadIdx.x + it * 32 * kAttnWarps;
      if (idx < N * D / 4) {
        kt[it] = reinterpret_cast<const float4*>(kb + (size_t)L * D)[idx];
        vt[it] = reinterpret_cast<const float4*>(vb + (size_t)L * D)[idx];
      }
    }
#pragma unroll
    for (int it = 0; it < QI; ++it) {
      const int idx = threadIdx.x + it * 32 * kAttnWarps;
      if (idx >= nmt * KS * 32) continue;
      const int ln = idx & 31, st = (idx >> 5) % KS, mt = (idx >> 5) / KS;
      uint4 ah, al;  // registers a0 (row g), a1 (row g+8), a2 (row g, +8 columns), a3 (row g+8, +8)
      split_h2(v[it][0], v[it][1], ah.x, al.x);
      split_h2(v[it][2], v[it][3], ah.y, al.y);
      split_h2(v[it][4], v[it][5], ah.z, al.z);
      split_h2(v[it][6], v[it][7], ah.w, al.w);
      uint4* dst = reinterpret_cast<uint4*>(Qf + ((size_t)(mt * KS + st) * 32 + ln) * 32);
      dst[0] = ah;
      dst[1] = al;
    }
#pragma unroll
    for (int it = 0; it < TI; ++it) {
      const int idx = threadIdx.x + it * 32 * kAttnWarps;
      if (idx < N * D / 4) {
        reinterpret_cast<float4*>(Kt)[idx] = kt[it];
        reinterpret_cast<float4*>(Vt)[idx] = vt[it];
      }
    }
  }
  consumers_sync();

  // values in the layout of the value product (warp w owns the dimension n-tiles
  // w*NTW .. w*NTW + NTW-1 of every query)
  float Or[MT][NTW][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int nn = 0; nn < NTW; ++nn)
#pragma unroll
      for (int e = 0; e < 4; ++e) Or[m][nn][e] = 0.0f;
  // Every tree slot holds one row for all the nodes that see it (a chain of several nodes,
  // say): then chunks reaching past the cache also take one B for all queries, the tree slots
  // reading that row (a key a query does not see is masked, a value it does not see has
  // weight zero).  Either way a row sees the same operations on the same values.
  bool merged = N > 1;
  for (int e = 0; e <= maxd; ++e) merged = merged && s_row[e] >= 0;
  bool ok = true;
  int n = 0;  // ring entries consumed
  for (int c = c_begin; c < c_end; ++c, n += 2) {
    const int eK = n % NE, eV = (n + 1) % NE;
    if (!consumers_all(mbar_wait(&full[eK], (n / NE) & 1))) {
      if (threadIdx.x == 0) atomicOr(&ctl->flags, FLAG_ERR_TIMEOUT);
      ok = false;  // a bounded wait expired: stop computing (uniform over the compute warps)
      break;
    }
    const float* Ks = reinterpret_cast<const float*>(ring_entry(eK));
    const float* Vs = reinterpret_cast<const float*>(ring_entry(eV));
    const int P0 = c * CH;
    const int jc = min(CH, L - P0);  // slots below jc come from the cache

    // ---- scores on the tensor cores: a score is the sum over 16-dimension steps of hi*hi +
    // hi*lo + lo*hi of the f16 splits of the query and the key, accumulated in f32 in that
    // fixed order (whichever warp computes it).
    {
      auto store = [&](const float (&acc)[4], int mt, int nt, int node) {
        // node < 0: every row; else only the rows of that node; keys 8nt + 2t, +1 as one float2
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int q = mt * 16 + lg + 8 * h;
          if (q >= QN || (node >= 0 && q / G != node)) continue;
          const int key = 8 * nt + 2 * lt;
          const int lim = L + s_dep[q / G] - P0;  // last slot of this chunk the query sees
          *reinterpret_cast<float2*>(SP + (size_t)q * SPS + key) =
              make_float2(key <= lim ? acc[2 * h] : -INFINITY, key + 1 <= lim ? acc[2 * h + 1] : -INFINITY);
        }
      };
      if (jc >= CH) {
        // every key of the chunk is cached: warp w takes m-tile w / WPM and the NTPW key n-tiles
        // from (w % WPM) * NTPW, one B per n-tile for all queries of the m-tile
        const int mw = warp / WPM, nt0 = (warp % WPM) * NTPW;
        if (mw < nmt) {
          float acc[NTPW][4];
#pragma unroll
          for (int i = 0; i < NTPW; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][e] = 0.0f;
#pragma unroll
          for (int st = 0; st < KS; ++st) {
            const uint4* af = reinterpret_cast<const uint4*>(Qf + ((size_t)(mw * KS + st) * 32 + lane) * 32);
            const uint4 ah = af[0], al = af[1];
#pragma unroll
            for (int i = 0; i < NTPW; ++i) {
              const float* kr = Ks + (size_t)(8 * (nt0 + i) + lg) * KSTR + st * 16 + 2 * lt;
              const float2 k0 = *reinterpret_cast<const float2*>(kr);
              const float2 k1 = *reinterpret_cast<const float2*>(kr + 8);
              uint32_t bh0, bl0, bh1, bl1;
              split_h2(k0.x, k0.y, bh0, bl0);
              split_h2(k1.x, k1.y, bh1, bl1);
              mma_split3(acc[i], ah, al, bh0, bh1, bl0, bl1);
            }
          }
#pragma unroll
          for (int i = 0; i < NTPW; ++i) store(acc[i], mw, nt0 + i, -1);
        }
      } else if (merged) {
        // chunk reaching past the cache with shared tree slots: the same partition, each lane's
        // key row from the cache, the shared tree row, or zero (past every node)
        const int mw = warp / WPM, nt0 = (warp % WPM) * NTPW;
        if (mw < nmt) {
          float acc[NTPW][4];
          const float* krow[NTPW];
#pragma unroll
          for (int i = 0; i < NTPW; ++i) {
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][e] = 0.0f;
            const int j = 8 * (nt0 + i) + lg;
            krow[i] = j < jc ? Ks + (size_t)j * KSTR
                             : (P0 + j - L <= maxd ? Kt + (size_t)s_row[P0 + j - L] * D : nullptr);
          }
#pragma unroll 1
          for (int st = 0; st < KS; ++st) {
            const uint4* af = reinterpret_cast<const uint4*>(Qf + ((size_t)(mw * KS + st) * 32 + lane) * 32);
            const uint4 ah = af[0], al = af[1];
#pragma unroll
            for (int i = 0; i < NTPW; ++i) {
              float2 k0 = make_float2(0.0f, 0.0f), k1 = make_float2(0.0f, 0.0f);
              if (krow[i] != nullptr) {
                k0 = *reinterpret_cast<const float2*>(krow[i] + st * 16 + 2 * lt);
                k1 = *reinterpret_cast<const float2*>(krow[i] + st * 16 + 2 * lt + 8);
              }
              uint32_t bh0, bl0, bh1, bl1;
              split_h2(k0.x, k0.y, bh0, bl0);
              split_h2(k1.x, k1.y, bh1, bl1);
              mma_split3(acc[i], ah, al, bh0, bh1, bl0, bl1);
            }
          }
#pragma unroll
          for (int i = 0; i < NTPW; ++i) store(acc[i], mw, nt0 + i, -1);
        }
      } else if (8 * warp + 7 < jc) {
        // chunk reaching past the cache, warp w takes key n-tile w for every m-tile; every key
        // of this n-tile is cached: one B for all queries
        const int j = 8 * warp + lg;  // key of this lane's B fragment
        float acc[MT][4];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[m][e] = 0.0f;
#pragma unroll 1
        for (int st = 0; st < KS; ++st) {
          const float* kr = Ks + (size_t)j * KSTR + st * 16 + 2 * lt;
          const float2 k0 = *reinterpret_cast<const float2*>(kr);
          const float2 k1 = *reinterpret_cast<const float2*>(kr + 8);
          uint32_t bh0, bl0, bh1, bl1;
          split_h2(k0.x, k0.y, bh0, bl0);
          split_h2(k1.x, k1.y, bh1, bl1);
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            if (m >= nmt) break;
            const uint4* af = reinterpret_cast<const uint4*>(Qf + ((size_t)(m * KS + st) * 32 + lane) * 32);
            mma_split3(acc[m], af[0], af[1], bh0, bh1, bl0, bl1);
          }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m)
          if (m < nmt) store(acc[m], m, warp, -1);
      } else {
        // n-tile w reaching past the cache: keys at L + e are each node's ancestors, so every
        // node takes its own B (cached keys are the same rows for all nodes); four nodes at a
        // time, each over the (at most MSPAN) m-tiles that hold its rows
        const int j = 8 * warp + lg;
        const int p = P0 + j;
        for (int nb = 0; nb < N; nb += 4) {
          const float* kr[4];
          int mlo[4], mcnt[4];  // first m-tile and m-tile count of each node (0: no node)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int node = nb + k;
            kr[k] = nullptr;
            mlo[k] = 0;
            mcnt[k] = 0;
            if (node < N) {
              if (j < jc) kr[k] = Ks + (size_t)j * KSTR;
              else if (p - L <= s_dep[node]) kr[k] = Kt + (size_t)s_path[node][p - L] * D;
              mlo[k] = (node * G) / 16;
              mcnt[k] = (node * G + G - 1) / 16 - mlo[k] + 1;
            }
          }
          float acc[4][MSPAN][4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int mi = 0; mi < MSPAN; ++mi)
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[k][mi][e] = 0.0f;
#pragma unroll 1
          for (int st = 0; st < KS; ++st) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              if (mcnt[k] == 0) continue;
              float2 k0 = make_float2(0.0f, 0.0f), k1 = make_float2(0.0f, 0.0f);
              if (kr[k] != nullptr) {
                k0 = *reinterpret_cast<const float2*>(kr[k] + st * 16 + 2 * lt);
                k1 = *reinterpret_cast<const float2*>(kr[k] + st * 16 + 2 * lt + 8);
              }
              uint32_t bh0, bl0, bh1, bl1;
              split_h2(k0.x, k0.y, bh0, bl0);
              split_h2(k1.x, k1.y, bh1, bl1);
#pragma unroll
              for (int mi = 0; mi < MSPAN; ++mi) {
                if (mi >= mcnt[k]) continue;
                const uint4* af =
                    reinterpret_cast<const uint4*>(Qf + ((size_t)((mlo[k] + mi) * KS + st) * 32 + lane) * 32);
                mma_split3(acc[k][mi], af[0], af[1], bh0, bh1, bl0, bl1);
              }
            }
          }
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int mi = 0; mi < MSPAN; ++mi)
              if (mi < mcnt[k]) store(acc[k][mi], mlo[k] + mi, warp, nb + k);
        }
      }
    }
    consumers_sync();
    if (threadIdx.x == 0) mbar_arrive(&empty[eK]);  // the key rows are no longer read
    if (!consumers_all(mbar_wait(&full[eV], ((n + 1) / NE) & 1))) {
      if (threadIdx.x == 0) atomicOr(&ctl->flags, FLAG_ERR_TIMEOUT);
      ok = false;
      break;
    }

    // ---- running statistics: warp w, queries w + 8u (interleaved); lane l holds slots 2l,
    // 2l+1.  The weights e go to the A fragments of the value product (f16 hi and lo): slot
    // pair (2l, 2l+1) is register (l & 4 ? 2 : 0) + (row >= 8) of fragment lane
    // 4 * (row & 7) + (l & 3), step l / 8, m-tile q / 16 (rows q and q + 8 of an m-tile
    // belong to the same warp).
    {
      float2 sv[QT];
      float mq[QT], mx[QT], l[QT], cs[QT], e0[QT], e1[QT];
      bool act[QT];
#pragma unroll
      for (int u = 0; u < QT; ++u) {
        const int q = warp + kAttnWarps * u;
        act[u] = q < QN && L + s_dep[min(q, QN - 1) / G] - P0 >= 0;  // the query sees this chunk
        sv[u] = make_float2(-INFINITY, -INFINITY);
        mq[u] = -INFINITY;
        if (act[u]) {
          sv[u] = *reinterpret_cast<const float2*>(SP + (size_t)q * SPS + 2 * lane);
          mq[u] = s_M[q];
        }
        mx[u] = fmaxf(sv[u].x, sv[u].y);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int u = 0; u < QT; ++u) mx[u] = fmaxf(mx[u], __shfl_xor_sync(0xffffffffu, mx[u], off));
#pragma unroll
      for (int u = 0; u < QT; ++u) {
        const float m = fmaxf(mq[u], mx[u]);
        mx[u] = m;
        cs[u] = 1.0f;
        e0[u] = e1[u] = 0.0f;
        if (act[u]) {
          cs[u] = (mq[u] == -INFINITY) ? 0.0f : expf(mq[u] - m);
          e0[u] = (sv[u].x == -INFINITY) ? 0.0f : expf(sv[u].x - m);
          e1[u] = (sv[u].y == -INFINITY) ? 0.0f : expf(sv[u].y - m);
        }
        l[u] = e0[u] + e1[u];
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int u = 0; u < QT; ++u) l[u] += __shfl_xor_sync(0xffffffffu, l[u], off);
      __syncwarp();
#pragma unroll
      for (int u = 0; u < QT; ++u) {
        const int q = warp + kAttnWarps * u;
        if (q >= QN) break;
        if (lane == 0) {
          if (act[u]) {
            s_L[q] = fmaf(s_L[q], cs[u], l[u]);
            s_M[q] = mx[u];
          }
          s_cs[q] = cs[u];
        }
        // the fragments hold 2^15 e (exact), so that small weights keep their low part in the
        // normal f16 range; the running values carry the same factor until they are stored
        uint32_t eh, el;
        split_h2(e0[u] * kAttnEScale, e1[u] * kAttnEScale, eh, el);
        const int r = q & 15;
        uint32_t* f = EF + ((size_t)((q >> 4) * VS + (lane >> 3)) * 32 + 4 * (r & 7) + (lane & 3)) * 8 +
                      ((lane & 4) ? 2 : 0) + (r >> 3);
        f[0] = eh;
        f[4] = el;
      }
    }
    consumers_sync();

    // ---- values on the tensor cores: O = O * c, then O += e . V for this warp's n-tiles,
    // 16-slot steps in order (rows past QN are never stored)
    {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m >= nmt) break;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float cq = s_cs[min(m * 16 + lg + ((e & 2) ? 8 : 0), QN - 1)];
#pragma unroll
          for (int nn = 0; nn < NTW; ++nn) Or[m][nn][e] *= cq;
        }
      }
      // B fragment of n-tile nn from slot rows r0..r3 (slots 2t, 2t+1, 2t+8, 2t+9 of the step);
      // a null row reads as zero
      auto vfrag = [&](const float* r0, const float* r1, const float* r2, const float* r3, int nn,
                       uint32_t& bh0, uint32_t& bl0, uint32_t& bh1, uint32_t& bl1) {
        const int dcol = (warp * NTW + nn) * 8 + lg;
        const float x0 = r0 ? r0[dcol] : 0.0f, x1 = r1 ? r1[dcol] : 0.0f;
        const float x2 = r2 ? r2[dcol] : 0.0f, x3 = r3 ? r3[dcol] : 0.0f;
        split_h2(x0, x1, bh0, bl0);
        split_h2(x2, x3, bh1, bl1);
      };
      // steps past the last slot that any node sees add nothing (their weights are zero); the
      // leading steps whose 16 slots are all cached (every step, when the tree slots are
      // shared) take one B for all queries
      const int nst = min(CH - 1, L + maxd - P0) / 16 + 1;
      const int ncs = min(nst, max(jc, 0) / 16);
#pragma unroll
      for (int st = 0; st < VS; ++st) {
        if (st < ncs) {
          const int js = st * 16 + 2 * lt;  // slots js, js+1, js+8, js+9 of this lane's B
          uint32_t bh0[NTW], bl0[NTW], bh1[NTW], bl1[NTW];
          const float* r0 = Vs + (size_t)js * VSTR;
#pragma unroll
          for (int nn = 0; nn < NTW; ++nn)
            vfrag(r0, r0 + VSTR, r0 + 8 * VSTR, r0 + 9 * VSTR, nn, bh0[nn], bl0[nn], bh1[nn], bl1[nn]);
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            if (m >= nmt) break;
            const uint4* af = reinterpret_cast<const uint4*>(EF + ((size_t)(m * VS + st) * 32 + lane) * 8);
            const uint4 ah = af[0], al = af[1];
#pragma unroll
            for (int nn = 0; nn < NTW; ++nn) mma_split3(Or[m][nn], ah, al, bh0[nn], bh1[nn], bl0[nn], bl1[nn]);
          }
        }
      }
      for (int st = ncs; st < nst; ++st) {
        const int js = st * 16 + 2 * lt;
        if (merged) {
          // shared tree slots: one B for all queries, rows from the cache, the shared tree row or
          // zero (past every node)
          auto vshared = [&](int jj) -> const float* {
            if (jj < jc) return Vs + (size_t)jj * VSTR;
            return P0 + jj - L <= maxd ? Vt + (size_t)s_row[P0 + jj - L] * D : nullptr;
          };
          const float* r0 = vshared(js);
          const float* r1 = vshared(js + 1);
          const float* r2 = vshared(js + 8);
          const float* r3 = vshared(js + 9);
          uint32_t bh0[NTW], bl0[NTW], bh1[NTW], bl1[NTW];
#pragma unroll
          for (int nn = 0; nn < NTW; ++nn) vfrag(r0, r1, r2, r3, nn, bh0[nn], bl0[nn], bh1[nn], bl1[nn]);
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            if (m >= nmt) break;
            const uint4* af = reinterpret_cast<const uint4*>(EF + ((size_t)(m * VS + st) * 32 + lane) * 8);
            const uint4 ah = af[0], al = af[1];
#pragma unroll
            for (int nn = 0; nn < NTW; ++nn) mma_split3(Or[m][nn], ah, al, bh0[nn], bh1[nn], bl0[nn], bl1[nn]);
          }
        } else {
          // per node: its own rows for the slots of this step (cache below jc, ancestors from
          // L on, zero past the node); four nodes at a time
          auto vrow = [&](int node, int kk) -> const float* {
            const int jj = js + (kk & 1) + ((kk & 2) ? 8 : 0);
            const int p = P0 + jj;
            if (jj < jc) return Vs + (size_t)jj * VSTR;
            if (p - L <= s_dep[node]) return Vt + (size_t)s_path[node][p - L] * D;
            return nullptr;
          };
          for (int nb = 0; nb < N; nb += 4) {
            const int nlast = min(N, nb + 4) - 1;
            const int glo = (nb * G) / 16, ghi = (nlast * G + G - 1) / 16;  // m-tiles of the group
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              if (m >= nmt) break;
              if (m < glo || m > ghi) continue;
              const uint4* af = reinterpret_cast<const uint4*>(EF + ((size_t)(m * VS + st) * 32 + lane) * 8);
              const uint4 ah = af[0], al = af[1];
#pragma unroll 1
              for (int k = 0; k < 4; ++k) {
                const int node = nb + k;
                if (node > nlast || m < (node * G) / 16 || m > (node * G + G - 1) / 16) continue;
                const float* r0 = vrow(node, 0);
                const float* r1 = vrow(node, 1);
                const float* r2 = vrow(node, 2);
                const float* r3 = vrow(node, 3);
#pragma unroll
                for (int nn = 0; nn < NTW; ++nn) {
                  uint32_t bh0, bl0, bh1, bl1;
                  vfrag(r0, r1, r2, r3, nn, bh0, bl0, bh1, bl1);
                  float d[4] = {Or[m][nn][0], Or[m][nn][1], Or[m][nn][2], Or[m][nn][3]};
                  mma_split3(d, ah, al, bh0, bh1, bl0, bl1);
                  // keep the rows of this node (the other rows take their own node's rows)
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const int q = m * 16 + lg + ((e & 2) ? 8 : 0);
                    if (q < QN && q / G == node) Or[m][nn][e] = d[e];
                  }
                }
              }
            }
          }
        }
      }
    }
    consumers_sync();
    if (threadIdx.x == 0) mbar_arrive(&empty[eV]);
  }
  // ---- this split's partial, then the merge by the last split of the head
  if (ok) {
#pragma unroll
    for (int u = 0; u < QT; ++u) {
      const int q = warp + kAttnWarps * u;
      if (q >= QN) break;
      if (L + s_dep[q / G] < c_begin * CH) continue;
      if (lane == 0) ml_part[((size_t)blockIdx.x * kMaxWidth + q / G) * Hq + kh * G + q % G] = make_float2(s_M[q], s_L[q]);
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m >= nmt) break;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int q = m * 16 + lg + 8 * h;
        if (q >= QN || L + s_dep[q / G] < c_begin * CH) continue;
        const size_t ob = ((size_t)blockIdx.x * kMaxWidth + q / G) * Hq + kh * G + q % G;
#pragma unroll
        for (int nn = 0; nn < NTW; ++nn)
          *reinterpret_cast<float2*>(o_part + ob * D + (warp * NTW + nn) * 8 + 2 * lt) =
              make_float2(Or[m][nn][2 * h] * (1.0f / kAttnEScale), Or[m][nn][2 * h + 1] * (1.0f / kAttnEScale));
      }
    }
  }
  if (!MERGE) return;
  consumers_sync();
  if (threadIdx.x == 0) {
    // release (after the barrier: this CTA's partials) and acquire (the other splits') at GPU
    // scope in one read-modify-write
    unsigned t;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(t) : "l"(tickets + kh) : "memory");
    const unsigned last = (t == (unsigned)(nsa - 1)) ? 1u : 0u;
    if (last) tickets[kh] = 0u;  // read again only by a later launch
    s_last = last;
  }
  consumers_sync();
  if (!s_last) return;
  const int d0 = lane * DL;  // merge: lane owns DL consecutive dimensions
  for (int q = warp; q < QN; q += kAttnWarps) {
    const int i = q / G, g = q % G;
    const int smax = ((L + s_dep[i]) / CH) / R;  // splits that saw this node
    const size_t hb = (size_t)i * Hq + kh * G + g;
    const size_t sstride = (size_t)kMaxWidth * Hq;
    float2 ml[8];
    float ov[8][DL];
    auto load_batch = [&](int sb) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (sb + k > smax) break;
        ml[k] = __ldcg(&ml_part[(sb + k) * sstride + hb]);
        const float* src = o_part + ((sb + k) * sstride + hb) * D + d0;
#pragma unroll
        for (int d = 0; d < DL; ++d) ov[k][d] = __ldcg(src + d);
      }
    };
    load_batch(0);  // in flight together with the loads of the maximum
    float M = -INFINITY;
    for (int s2 = lane; s2 <= smax; s2 += 32) M = fmaxf(M, __ldcg(&ml_part[s2 * sstride + hb].x));
    M = warp_max(M);
    float Ls = 0.0f, O[DL];
#pragma unroll
    for (int d = 0; d < DL; ++d) O[d] = 0.0f;
    for (int sb = 0; sb <= smax; sb += 8) {
      if (sb > 0) load_batch(sb);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (sb + k > smax) break;
        const float w = expf(ml[k].x - M);
        Ls = fmaf(w, ml[k].y, Ls);
#pragma unroll
        for (int d = 0; d < DL; ++d) O[d] = fmaf(w, ov[k][d], O[d]);
      }
    }
    float mx = 0.0f;
#pragma unroll
    for (int d = 0; d < DL; ++d) {
      const float res = __fdiv_rn(O[d], Ls);
      out[hb * D + d0 + d] = res;
      mx = fmaxf(mx, fabsf(res));
    }
    mx = warp_max(mx);
    if (lane == 0) mpart[hb] = make_float2(0.0f, mx);
  }
}

// Merge of the split partials for wide trees (defined in layers.cu).
__global__ void k_attn_merge(const SpecCtl* ctl, const TreeState* __restrict__ tree, const float* __restrict__ o_part,
                             const float2* __restrict__ ml_part, int Hq, int D, int R, int splits,
                             float* __restrict__ out, float2* __restrict__ mpart);

// Launch templates: every (G, QT) variant of head size D is configured up front; a launch picks
// the variant for N.
namespace {
// splits per KV head: about one CTA per SM (the ring holds two 64-position chunks)
inline int attn_splits(int Hkv) { return max(1, 148 / max(1, Hkv)); }

// attn_merge_inside(QT): the last split CTA merges small trees itself; wide trees (more than
// two queries per warp) merge in k_attn_merge, one CTA per (node, head)
constexpr bool attn_merge_inside(int QT) { return QT <= 2; }

template <int D, int G, int QT>
cudaError_t attn_launch(bool configure, size_t smem, const DecoderBufs& b, const ModelDims& m, int N, int layer,
                        cudaStream_t st) {
  constexpr bool MERGE = attn_merge_inside(QT);
  if (configure)
    return cudaFuncSetAttribute(k_attn<D, G, QT, MERGE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  const size_t lstride = (size_t)m.Hkv * b.kv_cap * m.D;
  const float* kc = b.kcache + layer * lstride;
  const float* vc = b.vcache + layer * lstride;
  const int splits = min(attn_splits(m.Hkv), b.n_chunks);
  const int R = (b.n_chunks + splits - 1) / splits;  // chunks per split (fixed per session)
  // more than kMaxWidth rows: a prefill bucket, N / kMaxWidth chains of kMaxWidth nodes (variants
  // that merge inside the kernel take one chain)
  const int nsub = N > kMaxWidth ? N / kMaxWidth : 1;
  const int Nn = N > kMaxWidth ? kMaxWidth : N;
  if (MERGE && nsub > 1) return cudaErrorInvalidValue;
  cudaError_t e = launch_pdl(k_attn<D, G, QT, MERGE>, dim3(splits, m.Hkv, nsub), dim3(kAttnThreads),
                             attn_smem_bytes(D, Nn * G), st, b.ctl, (const TreeState*)b.tree, Nn, (const float*)b.qrot,
                             kc, vc, b.kv_cap, m.Hq, R, b.o_part, (float2*)b.ml_part, b.attn_tickets, b.qkv, b.qpart,
                             b.tm_k, b.tm_v, layer);
  if (e != cudaSuccess || MERGE) return e;
  return launch_pdl(k_attn_merge, dim3(Nn * nsub, m.Hq), dim3(m.D), 0, st, (const SpecCtl*)b.ctl,
                    (const TreeState*)b.tree, (const float*)b.o_part, (const float2*)b.ml_part, m.Hq, m.D, R, splits,
                    b.qkv, b.qpart);
}
// QT: queries per compute warp, the power of two >= ceil(N*G / 8) (every variant is
// configured up front; launching picks the one for N)
template <int D, int G>
cudaError_t attn_dispatch(bool configure, size_t smem, const DecoderBufs& b, const ModelDims& m, int N, int layer,
                          cudaStream_t st) {
  constexpr int QTMAX = (kMaxWidth * G + kAttnWarps - 1) / kAttnWarps;
  const int Nn = N > kMaxWidth ? kMaxWidth : N;  // nodes per (sub-)chain
  const int qt = configure ? 1 : (Nn * G + kAttnWarps - 1) / kAttnWarps;
  cudaError_t e = cudaSuccess;
  if (configure || qt <= 1) e = attn_launch<D, G, 1>(configure, smem, b, m, N, layer, st);
  if constexpr (QTMAX > 1)
    if (e == cudaSuccess && (configure || (qt > 1 && qt <= 2))) e = attn_launch<D, G, 2>(configure, smem, b, m, N, layer, st);
  if constexpr (QTMAX > 2)
    if (e == cudaSuccess && (configure || (qt > 2 && qt <= 4))) e = attn_launch<D, G, 4>(configure, smem, b, m, N, layer, st);
  if constexpr (QTMAX > 4)
    if (e == cudaSuccess && (configure || (qt > 4 && qt <= 8))) e = attn_launch<D, G, 8>(configure, smem, b, m, N, layer, st);
  if constexpr (QTMAX > 8)
    if (e == cudaSuccess && (configure || qt > 8)) e = attn_launch<D, G, 16>(configure, smem, b, m, N, layer, st);
  return e;
}
template <int D>
cudaError_t attn_dispatch_g(int G, bool configure, size_t smem, const DecoderBufs& b, const ModelDims& m, int N,
                            int layer, cudaStream_t st) {
  switch (G) {
    case 1: return attn_dispatch<D, 1>(configure, smem, b, m, N, layer, st);
    case 2: return attn_dispatch<D, 2>(configure, smem, b, m, N, layer, st);
    case 3: return attn_dispatch<D, 3>(configure, smem, b, m, N, layer, st);
    case 4: return attn_dispatch<D, 4>(configure, smem, b, m, N, layer, st);
    case 5: return attn_dispatch<D, 5>(configure, smem, b, m, N, layer, st);
    case 6: return attn_dispatch<D, 6>(configure, smem, b, m, N, layer, st);
    case 7: return attn_dispatch<D, 7>(configure, smem, b, m, N, layer, st);
    case 8: return attn_dispatch<D, 8>(configure, smem, b, m, N, layer, st);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

// per head size, in its own translation unit
cudaError_t attn_dispatch_d64(int G, bool configure, size_t smem, const DecoderBufs& b, const ModelDims& m, int N,
                              int layer, cudaStream_t st);
cudaError_t attn_dispatch_d128(int G, bool configure, size_t smem, const DecoderBufs& b, const ModelDims& m, int N,
                               int layer, cudaStream_t st);

}  // namespace w4a8
