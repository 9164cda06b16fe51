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
//  * every per-token reduction (sum of squares, absmax) is a fixed per-thread sequence
//    followed by a fixed warp butterfly and a sequential sum of warp partials;
//  * attention chunks cover fixed logical positions [64c, 64c+64); a node at logical
//    position P sees positions <= P, taken from the cache below L_c and from its
//    ancestors' tree slots above; inside a chunk the dot products run over dimensions
//    in order, the softmax denominator is a fixed butterfly over the 64 slots and the
//    value sum runs over positions in order; chunks merge in ascending order.
#include "decoder.cuh"
#include "layers.cuh"

namespace w4a8 {

namespace {

__device__ __forceinline__ float block_sum_fixed(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = red[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) s += red[w];
  return s;
}

__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = red[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
  return m;
}

// Per-token int8 quantisation of K values val(k) (K % 32 == 0) straight into the matmul's
// activation fragments; also the group corrections and the token scale.
template <class F>
__device__ void quant_token(int t, int K, F val, float* red, uint4* af, float* corr, float* a_s) {
  float m = 0.0f;
  for (int k = threadIdx.x; k < K; k += blockDim.x) m = fmaxf(m, fabsf(val(k)));
  const float amax = block_max(m, red);
  const float s = __fdiv_rn(amax, 127.0f);
  const int nq = K / 4;
  const int Gp = groups_padded(K);
  for (int base = 0; base < nq; base += blockDim.x) {
    const int qd = base + threadIdx.x;
    const bool active = qd < nq;
    uint32_t codes = 0;
    int sum = 0;
    if (active) {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        int q = 0;
        if (s > 0.0f) q = (int)fminf(fmaxf(rintf(__fdiv_rn(val(4 * qd + b), s)), -127.0f), 127.0f);
        codes |= ((uint32_t)q & 0xffu) << (8 * b);
        sum += q;
      }
      afrag_store_quad(af, Gp, t, 4 * qd, codes);
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
    if (active && (threadIdx.x & 7) == 0) corr[(size_t)(qd >> 3) * 16 + t] = (float)sum * -0.015625f;
  }
  if (threadIdx.x == 0) a_s[t] = s;
}

__device__ __forceinline__ bool stopped(const SpecCtl* ctl) { return (ctl->flags & FLAG_STOP_MASK) != 0u; }

}  // namespace

// ------------------------------------------------------------------------------ embedding

__global__ void k_embed(SpecCtl* ctl, const TreeState* __restrict__ tree, int N, const uint32_t* __restrict__ ew,
                        const uint16_t* __restrict__ es, int H, int V, int kv_cap, float* __restrict__ x) {
  griddep_wait();
  if (stopped(ctl)) return;
  const int i = blockIdx.x;
  const int L = (int)ctl->committed_len;
  if (L + N > kv_cap) {
    if (i == 0 && threadIdx.x == 0) atomicOr(&ctl->flags, FLAG_ERR_CAPACITY);
    return;
  }
  const int tok = tree->tok[i];
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) atomicOr(&ctl->flags, FLAG_ERR_TOKEN);
    return;
  }
  const uint32_t* wr = ew + (size_t)tok * (H / 8);
  const uint16_t* sr = es + (size_t)tok * (H / 32);
  for (int w = threadIdx.x; w < H / 8; w += blockDim.x) {
    const uint32_t word = wr[w];
    const float s = __half2float(__ushort_as_half(sr[w >> 2]));
#pragma unroll
    for (int j = 0; j < 8; ++j) x[(size_t)i * H + 8 * w + j] = s * (float)((int)((word >> (4 * j)) & 15u) - 8);
  }
}

// --------------------------------------------------------------------- RMSNorm + quant

__global__ void k_rmsnorm_quant(const SpecCtl* ctl, const float* __restrict__ x, int H, float eps, uint4* af,
                                float* corr, float* a_s) {
  griddep_wait();
  if (stopped(ctl)) return;
  __shared__ float red[32];
  const int t = blockIdx.x;
  const float* xr = x + (size_t)t * H;
  float ss = 0.0f;
  for (int k = threadIdx.x; k < H; k += blockDim.x) ss = fmaf(xr[k], xr[k], ss);
  ss = block_sum_fixed(ss, red);
  const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)H), eps)));
  quant_token(t, H, [&](int k) { return xr[k] * r; }, red, af, corr, a_s);
}

// ------------------------------------------------------------------------- RoPE + KV

__global__ void k_rope_kv(const SpecCtl* ctl, const TreeState* __restrict__ tree, const float* __restrict__ qkv,
                          int Hq, int Hkv, int D, const float2* __restrict__ rope, float* kc, float* vc, int kv_cap,
                          float* __restrict__ qrot, float qscale) {
  griddep_wait();
  if (stopped(ctl)) return;
  const int i = blockIdx.x;
  const int L = (int)ctl->committed_len;
  const int pos = L + tree->depth[i];
  const int slot = L + i;
  const int half = D / 2;
  const int rows = (Hq + 2 * Hkv) * D;
  const float* row = qkv + (size_t)i * rows;
  const float2* cs = rope + (size_t)pos * half;
  for (int idx = threadIdx.x; idx < (Hq + Hkv) * half; idx += blockDim.x) {
    const int h = idx / half, j = idx % half;
    const float2 c = cs[j];
    const float a = row[h * D + j], b = row[h * D + j + half];
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
  for (int idx = threadIdx.x; idx < Hkv * D; idx += blockDim.x) {
    const int kh = idx / D, dd = idx % D;
    vc[((size_t)kh * kv_cap + slot) * D + dd] = row[(Hq + Hkv) * D + idx];
  }
}

// ---------------------------------------------------------------------- tree attention

template <int D>
__global__ void __launch_bounds__(256)
    k_attn_chunk(const SpecCtl* ctl, const TreeState* __restrict__ tree, int N, const float* __restrict__ qrot,
                 const float* __restrict__ kc, const float* __restrict__ vc, int kv_cap, int Hq, int Hkv,
                 float* __restrict__ o_part, float2* __restrict__ ml_part) {
  griddep_wait();
  if (stopped(ctl)) return;
  constexpr int CH = kAttnChunk;
  extern __shared__ float sm[];
  __shared__ int s_path[kMaxWidth][kMaxWidth];
  __shared__ int s_dep[kMaxWidth];
  const int c = blockIdx.x, kh = blockIdx.y, G = Hq / Hkv;
  const int L = (int)ctl->committed_len;
  const int P0 = c * CH;
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
  __syncthreads();
  int maxd = 0;
  for (int i = 0; i < N; ++i) maxd = max(maxd, s_dep[i]);
  if (P0 > L + maxd) return;
  const int ncache = max(0, min(CH, L - P0));
  const bool need_tree = P0 + CH > L;
  float* Ks = sm;
  float* Vs = Ks + CH * (D + 1);
  float* Kt = Vs + CH * D;
  float* Vt = Kt + kMaxWidth * (D + 1);
  float* Qs = Vt + kMaxWidth * D;
  const float* kb = kc + (size_t)kh * kv_cap * D;
  const float* vb = vc + (size_t)kh * kv_cap * D;
  for (int idx = threadIdx.x; idx < ncache * D; idx += blockDim.x) {
    const int r = idx / D, col = idx % D;
    Ks[r * (D + 1) + col] = kb[(size_t)(P0 + r) * D + col];
    Vs[r * D + col] = vb[(size_t)(P0 + r) * D + col];
  }
  if (need_tree) {
    for (int idx = threadIdx.x; idx < N * D; idx += blockDim.x) {
      const int r = idx / D, col = idx % D;
      Kt[r * (D + 1) + col] = kb[(size_t)(L + r) * D + col];
      Vt[r * D + col] = vb[(size_t)(L + r) * D + col];
    }
  }
  const int Nq = N * G;
  for (int idx = threadIdx.x; idx < Nq * D; idx += blockDim.x) {
    const int qi = idx / D, col = idx % D;
    const int i = qi / G, g = qi % G;
    Qs[qi * D + col] = qrot[((size_t)i * Hq + kh * G + g) * D + col];
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int qi = warp; qi < Nq; qi += blockDim.x >> 5) {
    const int i = qi / G, hq = kh * G + qi % G;
    const int pos = L + s_dep[i];
    if (pos < P0) continue;
    const float* q = Qs + qi * D;
    const int p0 = P0 + lane, p1 = P0 + lane + 32;
    const bool v0 = p0 <= pos, v1 = p1 <= pos;
    const float* k0 = v0 ? (p0 < L ? Ks + lane * (D + 1) : Kt + s_path[i][p0 - L] * (D + 1)) : Ks;
    const float* k1 = v1 ? (p1 < L ? Ks + (lane + 32) * (D + 1) : Kt + s_path[i][p1 - L] * (D + 1)) : Ks;
    float a0 = 0.0f, a1 = 0.0f;
#pragma unroll 8
    for (int k = 0; k < D; ++k) {
      const float qk = q[k];
      a0 = fmaf(qk, k0[k], a0);
      a1 = fmaf(qk, k1[k], a1);
    }
    const float s0 = v0 ? a0 : -INFINITY, s1 = v1 ? a1 : -INFINITY;
    const float m = warp_max(fmaxf(s0, s1));
    const float e0 = v0 ? expf(s0 - m) : 0.0f;
    const float e1 = v1 ? expf(s1 - m) : 0.0f;
    float l = e0 + e1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    float o_acc[D / 32];
#pragma unroll
    for (int r = 0; r < D / 32; ++r) o_acc[r] = 0.0f;
    const int last = min(CH - 1, pos - P0);
    for (int j = 0; j <= last; ++j) {
      const float e = __shfl_sync(0xffffffffu, j < 32 ? e0 : e1, j & 31);
      const int p = P0 + j;
      const float* vr = p < L ? Vs + j * D : Vt + s_path[i][p - L] * D;
#pragma unroll
      for (int r = 0; r < D / 32; ++r) o_acc[r] = fmaf(e, vr[lane + 32 * r], o_acc[r]);
    }
    const size_t ob = (((size_t)c * kMaxWidth + i) * Hq + hq);
#pragma unroll
    for (int r = 0; r < D / 32; ++r) o_part[ob * D + lane + 32 * r] = o_acc[r];
    if (lane == 0) ml_part[ob] = make_float2(m, l);
  }
}

__global__ void k_attn_merge_quant(const SpecCtl* ctl, const TreeState* __restrict__ tree,
                                   const float* __restrict__ o_part, const float2* __restrict__ ml_part, int Hq, int D,
                                   uint4* af, float* corr, float* a_s) {
  griddep_wait();
  if (stopped(ctl)) return;
  extern __shared__ float out[];
  __shared__ float red[32];
  const int i = blockIdx.x;
  const int L = (int)ctl->committed_len;
  const int pos = L + tree->depth[i];
  const int nc = pos / kAttnChunk + 1;
  for (int idx = threadIdx.x; idx < Hq * D; idx += blockDim.x) {
    const int h = idx / D, dd = idx % D;
    float M = -INFINITY;
    for (int c = 0; c < nc; ++c) M = fmaxf(M, ml_part[((size_t)c * kMaxWidth + i) * Hq + h].x);
    float Ls = 0.0f, O = 0.0f;
    for (int c = 0; c < nc; ++c) {
      const size_t b = ((size_t)c * kMaxWidth + i) * Hq + h;
      const float2 ml = ml_part[b];
      const float w = expf(ml.x - M);
      Ls = fmaf(w, ml.y, Ls);
      O = fmaf(w, o_part[b * D + dd], O);
    }
    out[idx] = __fdiv_rn(O, Ls);
  }
  __syncthreads();
  quant_token(i, Hq * D, [&](int k) { return out[k]; }, red, af, corr, a_s);
}

// ------------------------------------------------------------------------ SwiGLU + quant

__global__ void k_swiglu_quant(const SpecCtl* ctl, const float* __restrict__ gu, int F, uint4* af, float* corr,
                               float* a_s) {
  griddep_wait();
  if (stopped(ctl)) return;
  __shared__ float red[32];
  const int t = blockIdx.x;
  const float* g = gu + (size_t)t * 2 * F;
  const float* u = g + F;
  quant_token(t, F, [&](int k) {
    const float z = g[k];
    return __fdiv_rn(z, 1.0f + expf(-z)) * u[k];
  }, red, af, corr, a_s);
}

// -------------------------------------------------------------------------- argmax

__global__ void k_argmax(const SpecCtl* ctl, const float* __restrict__ logits, int V, int32_t* __restrict__ pred) {
  griddep_wait();
  if (stopped(ctl)) return;
  __shared__ float sv[32];
  __shared__ int si[32];
  const int t = blockIdx.x;
  const float* lr = logits + (size_t)t * V;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int k = threadIdx.x; k < V; k += blockDim.x) {
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
    if (bv == -INFINITY) bi = 0;
    pred[t] = bi;
  }
}

// ------------------------------------------------------------------------- launchers

size_t attn_smem_bytes(int D, int Nq) {
  return sizeof(float) * ((size_t)kAttnChunk * (D + 1) + (size_t)kAttnChunk * D + (size_t)kMaxWidth * (D + 1) +
                          (size_t)kMaxWidth * D + (size_t)Nq * D);
}

cudaError_t attn_configure(int D, size_t smem) {
  if (D == 64) return cudaFuncSetAttribute(k_attn_chunk<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (D == 128) return cudaFuncSetAttribute(k_attn_chunk<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return cudaErrorInvalidValue;
}

cudaError_t launch_embed(const DecoderBufs& b, const ModelDims& m, int N, const uint32_t* ew, const uint16_t* es,
                         cudaStream_t st) {
  return launch_pdl(k_embed, dim3(N), dim3(128), 0, st, b.ctl, (const TreeState*)b.tree, N, ew, es, m.H, m.V,
                    b.kv_cap, b.x);
}

cudaError_t launch_rmsnorm_quant(const DecoderBufs& b, const ModelDims& m, int N, cudaStream_t st) {
  return launch_pdl(k_rmsnorm_quant, dim3(N), dim3(256), 0, st, (const SpecCtl*)b.ctl, (const float*)b.x, m.H, m.eps,
                    b.af, b.corr, b.a_s);
}

cudaError_t launch_rope_kv(const DecoderBufs& b, const ModelDims& m, int N, int layer, cudaStream_t st) {
  const size_t lstride = (size_t)m.Hkv * b.kv_cap * m.D;
  const float qscale = (float)(1.0 / sqrt((double)m.D));
  return launch_pdl(k_rope_kv, dim3(N), dim3(256), 0, st, (const SpecCtl*)b.ctl, (const TreeState*)b.tree,
                    (const float*)b.qkv, m.Hq, m.Hkv, m.D, (const float2*)b.rope, b.kcache + layer * lstride,
                    b.vcache + layer * lstride, b.kv_cap, b.qrot, qscale);
}

cudaError_t launch_attention(const DecoderBufs& b, const ModelDims& m, int N, int layer, cudaStream_t st) {
  const size_t lstride = (size_t)m.Hkv * b.kv_cap * m.D;
  const int G = m.Hq / m.Hkv;
  const size_t smem = attn_smem_bytes(m.D, N * G);
  dim3 grid(b.n_chunks, m.Hkv);
  cudaError_t e;
  if (m.D == 64)
    e = launch_pdl(k_attn_chunk<64>, grid, dim3(256), smem, st, (const SpecCtl*)b.ctl, (const TreeState*)b.tree, N,
                   (const float*)b.qrot, (const float*)(b.kcache + layer * lstride),
                   (const float*)(b.vcache + layer * lstride), b.kv_cap, m.Hq, m.Hkv, b.o_part, (float2*)b.ml_part);
  else if (m.D == 128)
    e = launch_pdl(k_attn_chunk<128>, grid, dim3(256), smem, st, (const SpecCtl*)b.ctl, (const TreeState*)b.tree, N,
                   (const float*)b.qrot, (const float*)(b.kcache + layer * lstride),
                   (const float*)(b.vcache + layer * lstride), b.kv_cap, m.Hq, m.Hkv, b.o_part, (float2*)b.ml_part);
  else
    return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  return launch_pdl(k_attn_merge_quant, dim3(N), dim3(256), sizeof(float) * m.Hq * m.D, st, (const SpecCtl*)b.ctl,
                    (const TreeState*)b.tree, (const float*)b.o_part, (const float2*)b.ml_part, m.Hq, m.D, b.af,
                    b.corr, b.a_s);
}

cudaError_t launch_swiglu_quant(const DecoderBufs& b, const ModelDims& m, int N, cudaStream_t st) {
  return launch_pdl(k_swiglu_quant, dim3(N), dim3(256), 0, st, (const SpecCtl*)b.ctl, (const float*)b.gu, m.F, b.af,
                    b.corr, b.a_s);
}

cudaError_t launch_argmax(const DecoderBufs& b, const ModelDims& m, int N, cudaStream_t st) {
  return launch_pdl(k_argmax, dim3(N), dim3(1024), 0, st, (const SpecCtl*)b.ctl, (const float*)b.logits, m.V,
                    b.pred);
}

}  // namespace w4a8
