// Decoder kernels of one tree-verification pass (everything but the matmuls).
//
// "GPU-Resident Speculative Decoding ..." (Design > Small-Batch Verification Kernels):
// activation quantisation is fused into the RMSNorm and SiLU kernels that precede each
// matrix multiplication; attention splits the visible context into chunks that separate
// CTAs process and a second pass merges; the query heads that share a KV head read each
// key and value once.  (Design > GPU-Resident Speculation Loop): each node attends to the
// committed cache and to its ancestors.  (Implementation): the KV cache is fp32 and the
// reduction order is fixed, so a node's result does not depend on the tree around it.
//
// Order rules that make N-node verification bit-identical to N single-token steps:
//  * a per-token sum of squares is taken per 512-input slice (4 inputs per thread in order,
//    a warp butterfly, 4 warps in order) and the slices are added in order; maxima are exact;
//  * attention chunks cover fixed logical positions [64c, 64c+64); a node at logical
//    position P sees positions <= P, taken from the cache below L_c and from its
//    ancestors' tree slots above; inside a chunk the dot product of the key at slot j runs
//    over the dimensions starting at (j mod 32), the softmax denominator is a fixed
//    butterfly over the 64 slots and the value sum runs over positions in order; chunks
//    merge in ascending order.
#include "decoder.cuh"
#include "layers.cuh"

namespace w4a8 {

namespace {

constexpr int kQuantSlice = 512;  // inputs per CTA of the statistics and quantisation passes

__device__ __forceinline__ bool stopped(const SpecCtl* ctl) { return (ctl->flags & FLAG_STOP_MASK) != 0u; }

}  // namespace

// ------------------------------------------------------------------------------ embedding

__global__ void k_embed(SpecCtl* ctl, const TreeState* __restrict__ tree, int N, const uint32_t* __restrict__ ew,
                        const uint16_t* __restrict__ es, int H, int V, int kv_cap, float* __restrict__ x) {
  griddep_enter();
  if (stopped(ctl)) return;
  const int i = blockIdx.x;
  const int L = (int)ctl->committed_len;
  if (L + N > kv_cap) {
    if (i == 0 && blockIdx.y == 0 && threadIdx.x == 0) atomicOr(&ctl->flags, FLAG_ERR_CAPACITY);
    return;
  }
  const int tok = tree->tok[i];
  if (tok < 0 || tok >= V) {
    if (blockIdx.y == 0 && threadIdx.x == 0) atomicOr(&ctl->flags, FLAG_ERR_TOKEN);
    return;
  }
  const uint32_t* wr = ew + (size_t)tok * (H / 8);
  const uint16_t* sr = es + (size_t)tok * (H / 32);
  for (int w = blockIdx.y * blockDim.x + threadIdx.x; w < H / 8; w += blockDim.x * gridDim.y) {
    const uint32_t word = wr[w];
    const float s = __half2float(__ushort_as_half(sr[w >> 2]));
#pragma unroll
    for (int j = 0; j < 8; ++j) x[(size_t)i * H + 8 * w + j] = s * (float)((int)((word >> (4 * j)) & 15u) - 8);
  }
}

// --------------------------------------------------------------------- RMSNorm + quant

// Row statistics for RMSNorm, grid (token, slice of kQuantSlice inputs), 128 threads:
// per slice the sum of squares (each thread its 4 inputs in order, a warp butterfly, the
// 4 warps in order) and max |x|.
__global__ void k_row_stats(const SpecCtl* ctl, const float* __restrict__ x, int H, float2* __restrict__ part) {
  griddep_enter();
  if (stopped(ctl)) return;
  __shared__ float s_ss[4], s_mx[4];
  const int t = blockIdx.x, sl = blockIdx.y;
  const int k = sl * kQuantSlice + 4 * threadIdx.x;
  float ss = 0.0f, mx = 0.0f;
  if (k < H) {
    const float4 v = *reinterpret_cast<const float4*>(x + (size_t)t * H + k);
    ss = fmaf(v.x, v.x, ss); ss = fmaf(v.y, v.y, ss); ss = fmaf(v.z, v.z, ss); ss = fmaf(v.w, v.w, ss);
    mx = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ss += __shfl_xor_sync(0xffffffffu, ss, o);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if ((threadIdx.x & 31) == 0) { s_ss[threadIdx.x >> 5] = ss; s_mx[threadIdx.x >> 5] = mx; }
  __syncthreads();
  if (threadIdx.x == 0)
    part[(size_t)t * gridDim.y + sl] = make_float2(((s_ss[0] + s_ss[1]) + s_ss[2]) + s_ss[3],
                                                   fmaxf(fmaxf(s_mx[0], s_mx[1]), fmaxf(s_mx[2], s_mx[3])));
}

// Quantisation pass, grid (token, slice), 128 threads, one 4-input quad per thread.  The
// per-token scale comes from the slice partials (fixed order): mode 0 plain (amax = max of
// the partial maxima), mode 1 RMSNorm (x scaled by r = 1/sqrt(sum of squares / K + eps), and
// amax = max |x| * r, equal to the maximum of the rounded products since rounding is monotone).
template <int MODE>
__global__ void k_quant_slices(const SpecCtl* ctl, const float* __restrict__ x, int K, int ldx,
                               const float2* __restrict__ part, int nparts, float eps, uint8_t* act, int M,
                               float* a_s) {
  griddep_enter();
  if (stopped(ctl)) return;
  const int t = blockIdx.x, sl = blockIdx.y;
  float mx = 0.0f, r = 1.0f;
  if (MODE == 1) {
    float ss = 0.0f;
    for (int p = 0; p < nparts; ++p) {
      const float2 v = part[(size_t)t * nparts + p];
      ss = ss + v.x;
      mx = fmaxf(mx, v.y);
    }
    r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)K), eps)));
    mx = mx * r;
  } else {
    for (int p = 0; p < nparts; ++p) mx = fmaxf(mx, part[(size_t)t * nparts + p].y);
  }
  const float s = __fdiv_rn(mx, 127.0f);
  const int NT = act_tiles(M);
  const int k = sl * kQuantSlice + 4 * threadIdx.x;
  const bool active = k < K;  // K % 32 == 0: groups of 8 lanes are all active or all idle
  const bool pad = !active && k < chunks_of(K) * 64;  // the zero group that completes the last chunk
  uint32_t codes = 0;
  int sum = 0;
  if (active) {
    float4 v = *reinterpret_cast<const float4*>(x + (size_t)t * ldx + k);
    if (MODE == 1) { v.x = v.x * r; v.y = v.y * r; v.z = v.z * r; v.w = v.w * r; }
    const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      int q = 0;
      if (s > 0.0f) q = (int)fminf(fmaxf(rintf(__fdiv_rn(vv[b], s)), -127.0f), 127.0f);
      codes |= ((uint32_t)q & 0xffu) << (8 * b);
      sum += q;
    }
  }
  if (active || pad) act_store_quad(act, NT, t, k, codes);
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  sum += __shfl_xor_sync(0xffffffffu, sum, 4);
  if ((active || pad) && (threadIdx.x & 7) == 0) act_store_corr(act, NT, t, k >> 5, sum);
  if (sl == 0 && threadIdx.x == 0) a_s[t] = s;
}

// ------------------------------------------------------------------------- RoPE + KV

// grid (node, head among Hq query + Hkv key + Hkv value heads), D/2 threads
__global__ void k_rope_kv(const SpecCtl* ctl, const TreeState* __restrict__ tree, const float* __restrict__ qkv,
                          int Hq, int Hkv, int D, const float2* __restrict__ rope, float* kc, float* vc, int kv_cap,
                          float* __restrict__ qrot, float qscale) {
  griddep_enter();
  if (stopped(ctl)) return;
  const int i = blockIdx.x, h = blockIdx.y, j = threadIdx.x;
  const int L = (int)ctl->committed_len;
  const int pos = L + tree->depth[i];
  const int slot = L + i;
  const int half = D / 2;
  const float* row = qkv + (size_t)i * (Hq + 2 * Hkv) * D + (size_t)h * D;
  if (h >= Hq + Hkv) {  // value head: plain copy into the cache
    float* vr = vc + ((size_t)(h - Hq - Hkv) * kv_cap + slot) * D;
    vr[j] = row[j];
    vr[j + half] = row[j + half];
    return;
  }
  const float2 c = rope[(size_t)pos * half + j];
  const float a = row[j], b = row[j + half];
  const float o1 = a * c.x - b * c.y;
  const float o2 = b * c.x + a * c.y;
  if (h < Hq) {
    qrot[((size_t)i * Hq + h) * D + j] = o1 * qscale;
    qrot[((size_t)i * Hq + h) * D + j + half] = o2 * qscale;
  } else {
    float* kr = kc + ((size_t)(h - Hq) * kv_cap + slot) * D;
    kr[j] = o1;
    kr[j + half] = o2;
  }
}

// ---------------------------------------------------------------------- tree attention

// Chunk pass, grid (chunk of kAttnChunk logical positions, KV head).  A warp task is (tree node,
// GW of the G query heads of the KV head); warps take tasks round-robin (GW = G for wide trees,
// GW = 1 when N * G <= 8 so that small trees still use several warps).  The chunk's cached K and V rows (contiguous)
// and the tree rows are fetched with cp.async.bulk.  A warp scores the keys of its node for all
// G query heads of the KV head at once (each key and value read serves G queries); lane j takes
// the keys at chunk slots j and j+32.  The dot product of the key at slot j runs over the
// dimensions starting at (j mod 32) and wrapping (conflict-free shared-memory reads); the
// value sum of a (head, dimension) runs over positions in order.  Every order is a function of
// the logical position only.
template <int D, int G, int GW>
__global__ void __launch_bounds__(256)
    k_attn_chunk(SpecCtl* ctl, const TreeState* __restrict__ tree, int N, const float* __restrict__ qrot,
                 const float* __restrict__ kc, const float* __restrict__ vc, int kv_cap, int Hq,
                 float* __restrict__ o_part, float2* __restrict__ ml_part) {
  griddep_enter();
  if (stopped(ctl)) return;
  constexpr int CH = kAttnChunk;
  constexpr int R = D / 32;
  extern __shared__ __align__(128) float sm[];
  __shared__ int s_path[kMaxWidth][kMaxWidth];
  __shared__ int s_dep[kMaxWidth];
  __shared__ uint64_t bar;
  const int c = blockIdx.x, kh = blockIdx.y;
  const int L = (int)ctl->committed_len;
  const int P0 = c * CH;
  int maxd = 0;
  for (int i = 0; i < N; ++i) maxd = max(maxd, tree->depth[i]);
  if (P0 > L + maxd) return;  // uniform over the CTA
  const int ncache = max(0, min(CH, L - P0));
  const bool need_tree = P0 + CH > L;
  float* Ks = sm;
  float* Vs = Ks + CH * D;
  float* Kt = Vs + CH * D;
  float* Vt = Kt + kMaxWidth * D;
  float* Qs = Vt + kMaxWidth * D;  // [node][G][D]
  const float* kb = kc + (size_t)kh * kv_cap * D;
  const float* vb = vc + (size_t)kh * kv_cap * D;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    mbar_expect_tx(&bar, (unsigned)((ncache + (need_tree ? N : 0)) * D * 4 * 2));
    if (ncache > 0) {
      bulk_g2s(Ks, kb + (size_t)P0 * D, (unsigned)(ncache * D * 4), &bar);
      bulk_g2s(Vs, vb + (size_t)P0 * D, (unsigned)(ncache * D * 4), &bar);
    }
    if (need_tree) {
      bulk_g2s(Kt, kb + (size_t)L * D, (unsigned)(N * D * 4), &bar);
      bulk_g2s(Vt, vb + (size_t)L * D, (unsigned)(N * D * 4), &bar);
    }
  }
  if (threadIdx.x < N) {
    const int i = threadIdx.x;
    const int d = tree->depth[i];
    s_dep[i] = d;
    int cur = i;
    for (int e = d; e >= 0; --e) {
      s_path[i][e] = cur;
      cur = e > 0 ? tree->parent[cur] : 0;
    }
  }
  // queries of the CTA's nodes: the G heads of KV head kh are consecutive in qrot
  for (int idx = threadIdx.x; idx < N * G * D / 4; idx += blockDim.x) {
    const int i = (4 * idx) / (G * D), rem = (4 * idx) % (G * D);
    *reinterpret_cast<float4*>(Qs + (size_t)i * G * D + rem) =
        *reinterpret_cast<const float4*>(qrot + ((size_t)i * Hq + kh * G) * D + rem);
  }
  __syncthreads();  // barrier initialised, paths and queries in place
  const int ok = __syncthreads_and(mbar_wait(&bar, 0) ? 1 : 0);
  if (!ok) {  // a bounded wait expired: report and skip the chunk
    if (threadIdx.x == 0) atomicOr(&ctl->flags, FLAG_ERR_TIMEOUT);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int NS = G / GW;  // head subsets per node
  for (int task = warp; task < N * NS; task += blockDim.x >> 5) {
    const int i = task / NS, hs = task % NS;
    const int pos = L + s_dep[i];
    if (pos < P0) continue;
    const float* q = Qs + ((size_t)i * G + hs * GW) * D;
    const int p0 = P0 + lane, p1 = P0 + lane + 32;
    const bool v0 = p0 <= pos, v1 = p1 <= pos;
    const float* k0 = v0 ? (p0 < L ? Ks + lane * D : Kt + s_path[i][p0 - L] * D) : Ks;
    const float* k1 = v1 ? (p1 < L ? Ks + (lane + 32) * D : Kt + s_path[i][p1 - L] * D) : Ks;
    float a0[GW], a1[GW];
#pragma unroll
    for (int g = 0; g < GW; ++g) a0[g] = a1[g] = 0.0f;
#pragma unroll 8
    for (int kk = 0; kk < D; ++kk) {
      const int k = (kk + lane) & (D - 1);
      const float x0 = k0[k], x1 = k1[k];
#pragma unroll
      for (int g = 0; g < GW; ++g) {
        const float qk = q[g * D + k];
        a0[g] = fmaf(qk, x0, a0[g]);
        a1[g] = fmaf(qk, x1, a1[g]);
      }
    }
    float e0[GW], e1[GW], mg[GW], lg[GW];
#pragma unroll
    for (int g = 0; g < GW; ++g) {
      const float s0 = v0 ? a0[g] : -INFINITY, s1 = v1 ? a1[g] : -INFINITY;
      mg[g] = warp_max(fmaxf(s0, s1));
      e0[g] = v0 ? expf(s0 - mg[g]) : 0.0f;
      e1[g] = v1 ? expf(s1 - mg[g]) : 0.0f;
      float l = e0[g] + e1[g];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      lg[g] = l;
    }
    float o_acc[GW][R];
#pragma unroll
    for (int g = 0; g < GW; ++g)
#pragma unroll
      for (int r = 0; r < R; ++r) o_acc[g][r] = 0.0f;
    const int last = min(CH - 1, pos - P0);
    for (int j = 0; j <= last; ++j) {
      const int p = P0 + j;
      const float* vr = p < L ? Vs + j * D : Vt + s_path[i][p - L] * D;
      float vv[R];
#pragma unroll
      for (int r = 0; r < R; ++r) vv[r] = vr[lane + 32 * r];
#pragma unroll
      for (int g = 0; g < GW; ++g) {
        const float e = __shfl_sync(0xffffffffu, j < 32 ? e0[g] : e1[g], j & 31);
#pragma unroll
        for (int r = 0; r < R; ++r) o_acc[g][r] = fmaf(e, vv[r], o_acc[g][r]);
      }
    }
#pragma unroll
    for (int g = 0; g < GW; ++g) {
      const size_t ob = (((size_t)c * kMaxWidth + i) * Hq + kh * G + hs * GW + g);
#pragma unroll
      for (int r = 0; r < R; ++r) o_part[ob * D + lane + 32 * r] = o_acc[g][r];
      if (lane == 0) ml_part[ob] = make_float2(mg[g], lg[g]);
    }
  }
}

// Merge of the chunk partials: grid (node, query head), one thread per dimension; chunks in
// ascending order (M = max m_c; L = sum exp(m_c - M) l_c; O = sum exp(m_c - M) o_c).
__global__ void k_attn_merge(const SpecCtl* ctl, const TreeState* __restrict__ tree, const float* __restrict__ o_part,
                             const float2* __restrict__ ml_part, int Hq, int D, float* __restrict__ out,
                             float2* __restrict__ mpart) {
  griddep_enter();
  if (stopped(ctl)) return;
  const int i = blockIdx.x, h = blockIdx.y, dd = threadIdx.x;
  const int L = (int)ctl->committed_len;
  const int pos = L + tree->depth[i];
  const int nc = pos / kAttnChunk + 1;
  const size_t stride = (size_t)kMaxWidth * Hq;  // ml entries between consecutive chunks
  const float2* ml = ml_part + (size_t)i * Hq + h;
  const float* op = o_part + ((size_t)i * Hq + h) * D + dd;
  float M = -INFINITY;
  for (int c = 0; c < nc; ++c) M = fmaxf(M, ml[c * stride].x);
  float Ls = 0.0f, O = 0.0f;
  int c = 0;
  for (; c + 8 <= nc; c += 8) {
    float2 m8[8];
    float o8[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      m8[q] = ml[(c + q) * stride];
      o8[q] = op[(size_t)(c + q) * stride * D];
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float w = expf(m8[q].x - M);
      Ls = fmaf(w, m8[q].y, Ls);
      O = fmaf(w, o8[q], O);
    }
  }
  for (; c < nc; ++c) {
    const float2 m1 = ml[c * stride];
    const float w = expf(m1.x - M);
    Ls = fmaf(w, m1.y, Ls);
    O = fmaf(w, op[(size_t)c * stride * D], O);
  }
  const float res = __fdiv_rn(O, Ls);
  out[((size_t)i * Hq + h) * D + dd] = res;
  __shared__ float s_mx[4];
  const float mx = warp_max(fabsf(res));
  if ((dd & 31) == 0) s_mx[dd >> 5] = mx;
  __syncthreads();
  if (dd == 0) {
    float m = s_mx[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, s_mx[w]);
    mpart[(size_t)i * Hq + h] = make_float2(0.0f, m);
  }
}

// ------------------------------------------------------------------------ SwiGLU

// grid (token, slice of kQuantSlice), 128 threads: h = silu(gate) * up written over the gate
// half of the gate|up buffer, and the slice maximum of |h|.
__global__ void k_swiglu(const SpecCtl* ctl, float* __restrict__ gu, int F, float2* __restrict__ part) {
  griddep_enter();
  if (stopped(ctl)) return;
  __shared__ float s_mx[4];
  const int t = blockIdx.x, sl = blockIdx.y;
  const int k = sl * kQuantSlice + 4 * threadIdx.x;
  float mx = 0.0f;
  if (k < F) {
    float* g = gu + (size_t)t * 2 * F + k;
    const float4 gv = *reinterpret_cast<const float4*>(g);
    const float4 uv = *reinterpret_cast<const float4*>(g + F);
    float4 h;
    h.x = __fdiv_rn(gv.x, 1.0f + expf(-gv.x)) * uv.x;
    h.y = __fdiv_rn(gv.y, 1.0f + expf(-gv.y)) * uv.y;
    h.z = __fdiv_rn(gv.z, 1.0f + expf(-gv.z)) * uv.z;
    h.w = __fdiv_rn(gv.w, 1.0f + expf(-gv.w)) * uv.w;
    *reinterpret_cast<float4*>(g) = h;
    mx = fmaxf(fmaxf(fabsf(h.x), fabsf(h.y)), fmaxf(fabsf(h.z), fabsf(h.w)));
  }
  mx = warp_max(mx);
  if ((threadIdx.x & 31) == 0) s_mx[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0)
    part[(size_t)t * gridDim.y + sl] = make_float2(0.0f, fmaxf(fmaxf(s_mx[0], s_mx[1]), fmaxf(s_mx[2], s_mx[3])));
}

// -------------------------------------------------------------------------- argmax

constexpr int kArgmaxSlice = 8192;

// grid (token, slice of kArgmaxSlice logits): slice maxima (ties -> lowest index), then the
// last CTA of the token to finish (ticket) reduces the slice partials.
__global__ void k_argmax(const SpecCtl* ctl, const float* __restrict__ logits, int V, float2* __restrict__ part,
                         unsigned* __restrict__ tickets, int32_t* __restrict__ pred) {
  griddep_enter();
  if (stopped(ctl)) return;
  __shared__ float sv[32];
  __shared__ int si[32];
  __shared__ unsigned s_ticket;
  const int t = blockIdx.x, sl = blockIdx.y, ns = gridDim.y;
  const float* lr = logits + (size_t)t * V;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  const int k1 = min(V, (sl + 1) * kArgmaxSlice);
  for (int k = sl * kArgmaxSlice + threadIdx.x; k < k1; k += blockDim.x) {
    const float v = lr[k];
    if (v > bv) { bv = v; bi = k; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
  }
  if ((threadIdx.x & 31) == 0) { sv[threadIdx.x >> 5] = bv; si[threadIdx.x >> 5] = bi; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
      if (sv[w] > bv || (sv[w] == bv && si[w] < bi)) { bv = sv[w]; bi = si[w]; }
    part[t * ns + sl] = make_float2(bv, __int_as_float(bi));
    __threadfence();
    s_ticket = atomicAdd(tickets + t, 1u);
    if (s_ticket == (unsigned)(ns - 1)) {
      __threadfence();
      float v = -INFINITY;
      int ix = 0x7fffffff;
      for (int q = 0; q < ns; ++q) {
        const float2 pq = __ldcg(part + t * ns + q);
        const int iq = __float_as_int(pq.y);
        if (pq.x > v || (pq.x == v && iq < ix)) { v = pq.x; ix = iq; }
      }
      pred[t] = (v == -INFINITY) ? 0 : ix;
      tickets[t] = 0u;
    }
  }
}

// ------------------------------------------------------------------------- launchers

size_t attn_smem_bytes(int D, int Nq) {
  return sizeof(float) * ((size_t)2 * kAttnChunk * D + (size_t)2 * kMaxWidth * D + (size_t)Nq * D);
}

namespace {
template <int D, int G>
cudaError_t attn_dispatch(bool configure, size_t smem, const DecoderBufs& b, const ModelDims& m, int N, int layer,
                          cudaStream_t st) {
  if (configure) {
    cudaError_t e = cudaFuncSetAttribute(k_attn_chunk<D, G, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_attn_chunk<D, G, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  }
  const size_t lstride = (size_t)m.Hkv * b.kv_cap * m.D;
  const float* kc = b.kcache + layer * lstride;
  const float* vc = b.vcache + layer * lstride;
  if (N * G <= 8)  // small trees: one warp per (node, head)
    return launch_pdl(k_attn_chunk<D, G, 1>, dim3(b.n_chunks, m.Hkv), dim3(32 * N * G), smem, st, b.ctl,
                      (const TreeState*)b.tree, N, (const float*)b.qrot, kc, vc, b.kv_cap, m.Hq, b.o_part,
                      (float2*)b.ml_part);
  return launch_pdl(k_attn_chunk<D, G, G>, dim3(b.n_chunks, m.Hkv), dim3(32 * (N < 8 ? N : 8)), smem, st, b.ctl,
                    (const TreeState*)b.tree, N, (const float*)b.qrot, kc, vc, b.kv_cap, m.Hq, b.o_part,
                    (float2*)b.ml_part);
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
cudaError_t attn_any(int D, int G, bool configure, size_t smem, const DecoderBufs& b, const ModelDims& m, int N,
                     int layer, cudaStream_t st) {
  if (D == 64) return attn_dispatch_g<64>(G, configure, smem, b, m, N, layer, st);
  if (D == 128) return attn_dispatch_g<128>(G, configure, smem, b, m, N, layer, st);
  return cudaErrorInvalidValue;
}
}  // namespace

cudaError_t attn_configure(const ModelDims& m, size_t smem) {
  DecoderBufs b{};
  return attn_any(m.D, m.Hq / m.Hkv, true, smem, b, m, 1, 0, nullptr);
}

cudaError_t launch_embed(const DecoderBufs& b, const ModelDims& m, int N, const uint32_t* ew, const uint16_t* es,
                         cudaStream_t st) {
  return launch_pdl(k_embed, dim3(N, (m.H / 8 + 127) / 128), dim3(128), 0, st, b.ctl, (const TreeState*)b.tree, N, ew,
                    es, m.H, m.V,
                    b.kv_cap, b.x);
}

cudaError_t launch_rmsnorm_quant(const DecoderBufs& b, const ModelDims& m, int N, cudaStream_t st) {
  const int ns = (m.H + kQuantSlice - 1) / kQuantSlice;
  cudaError_t e = launch_pdl(k_row_stats, dim3(N, ns), dim3(kQuantSlice / 4), 0, st, (const SpecCtl*)b.ctl,
                             (const float*)b.x, m.H, b.qpart);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_quant_slices<1>, dim3(N, ns), dim3(kQuantSlice / 4), 0, st, (const SpecCtl*)b.ctl,
                    (const float*)b.x, m.H, m.H, (const float2*)b.qpart, ns, m.eps, b.act, N, b.a_s);
}

cudaError_t launch_rope_kv(const DecoderBufs& b, const ModelDims& m, int N, int layer, cudaStream_t st) {
  const size_t lstride = (size_t)m.Hkv * b.kv_cap * m.D;
  const float qscale = (float)(1.0 / sqrt((double)m.D));
  return launch_pdl(k_rope_kv, dim3(N, m.Hq + 2 * m.Hkv), dim3(m.D / 2), 0, st, (const SpecCtl*)b.ctl,
                    (const TreeState*)b.tree,
                    (const float*)b.qkv, m.Hq, m.Hkv, m.D, (const float2*)b.rope, b.kcache + layer * lstride,
                    b.vcache + layer * lstride, b.kv_cap, b.qrot, qscale);
}

cudaError_t launch_attention(const DecoderBufs& b, const ModelDims& m, int N, int layer, cudaStream_t st) {
  const int G = m.Hq / m.Hkv;
  cudaError_t e = attn_any(m.D, G, false, attn_smem_bytes(m.D, N * G), b, m, N, layer, st);
  if (e != cudaSuccess) return e;
  e = launch_pdl(k_attn_merge, dim3(N, m.Hq), dim3(m.D), 0, st, (const SpecCtl*)b.ctl, (const TreeState*)b.tree,
                 (const float*)b.o_part, (const float2*)b.ml_part, m.Hq, m.D, b.qkv, b.qpart);
  if (e != cudaSuccess) return e;
  // the attention output (in the qkv buffer, [N][Hq*D]) -> int8 fragments of the O projection
  const int QD = m.Hq * m.D;
  return launch_pdl(k_quant_slices<0>, dim3(N, (QD + kQuantSlice - 1) / kQuantSlice), dim3(kQuantSlice / 4), 0, st,
                    (const SpecCtl*)b.ctl, (const float*)b.qkv, QD, QD, (const float2*)b.qpart, m.Hq, 0.0f, b.act, N,
                    b.a_s);
}

cudaError_t launch_swiglu_quant(const DecoderBufs& b, const ModelDims& m, int N, cudaStream_t st) {
  const int ns = (m.F + kQuantSlice - 1) / kQuantSlice;
  cudaError_t e = launch_pdl(k_swiglu, dim3(N, ns), dim3(kQuantSlice / 4), 0, st, (const SpecCtl*)b.ctl, b.gu, m.F,
                             b.qpart);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_quant_slices<0>, dim3(N, ns), dim3(kQuantSlice / 4), 0, st, (const SpecCtl*)b.ctl,
                    (const float*)b.gu, m.F, 2 * m.F, (const float2*)b.qpart, ns, 0.0f, b.act, N, b.a_s);
}

cudaError_t launch_argmax(const DecoderBufs& b, const ModelDims& m, int N, cudaStream_t st) {
  return launch_pdl(k_argmax, dim3(N, (m.V + kArgmaxSlice - 1) / kArgmaxSlice), dim3(512), 0, st,
                    (const SpecCtl*)b.ctl, (const float*)b.logits, m.V, b.argmax_part, b.argmax_tickets, b.pred);
}

}  // namespace w4a8
