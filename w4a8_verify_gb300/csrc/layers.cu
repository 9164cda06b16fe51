// Decoder kernels of one tree-verification pass other than the matmuls and the tree
// attention (attention.cuh): embedding, RMSNorm statistics and activation quantisation, RoPE
// and KV write, SwiGLU, the attention merge for wide trees, argmax, and their launchers.
//
// "GPU-Resident Speculative Decoding ..." (Design > Small-Batch Verification Kernels):
// activation quantisation is fused into the RMSNorm and SiLU kernels that precede each
// matrix multiplication.  (Implementation): the KV cache is fp32 and the reduction order is
// fixed, so a node's result does not depend on the tree around it.
//
// Order rules that make N-node verification bit-identical to N single-token steps:
//  * a per-token sum of squares is taken per 512-input slice (4 inputs per thread in order,
//    a warp butterfly, 4 warps in order) and the slices are added in order; maxima are exact;
//  * split-K partial outputs of the projections are folded in ascending slice order;
//  * attention: see attention.cuh (chunks of fixed logical positions, tensor-core products
//    whose order depends on the logical position only, splits merged in ascending order).
#include "attention.cuh"
#include "layers.cuh"

namespace w4a8 {

namespace {

constexpr int kQuantSlice = 512;  // inputs per CTA of the statistics and quantisation passes


}  // namespace

// ------------------------------------------------------------------------------ embedding

// Token i of the pass: tree node i, or (chain != nullptr: a prefill bucket) context token
// committed_len + i.
__global__ void k_embed(SpecCtl* ctl, const TreeState* __restrict__ tree, const int32_t* __restrict__ chain, int N,
                        const uint32_t* __restrict__ ew, const uint16_t* __restrict__ es, int H, int V, int kv_cap,
                        float* __restrict__ x) {
  griddep_enter();
  if (stopped(ctl)) return;
  const int i = blockIdx.x;
  const int L = (int)ctl->committed_len;
  if (L + N > kv_cap) {
    if (i == 0 && blockIdx.y == 0 && threadIdx.x == 0) atomicOr(&ctl->flags, FLAG_ERR_CAPACITY);
    return;
  }
  const int tok = chain != nullptr ? chain[L + i] : tree->tok[i];
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
__global__ void __launch_bounds__(kQuantSlice / 4)
    k_row_stats(const SpecCtl* ctl, float* __restrict__ x, int H, float2* __restrict__ part,
                            const float* __restrict__ res, int res_S, const float* __restrict__ res_as) {
  griddep_enter();
  if (stopped(ctl)) return;
  __shared__ float s_ss[4], s_mx[4];
  const int t = blockIdx.x, sl = blockIdx.y;
  const int k = sl * kQuantSlice + 4 * threadIdx.x;
  float ss = 0.0f, mx = 0.0f;
  if (k < H) {
    float4 v = *reinterpret_cast<const float4*>(x + (size_t)t * H + k);
    if (res != nullptr) {  // residual update by the preceding projection (its slices folded here)
      const float4 r = mm_fold4(res, res_S, H, t, k, res_as);
      v.x = v.x + r.x;
      v.y = v.y + r.y;
      v.z = v.z + r.z;
      v.w = v.w + r.w;
      *reinterpret_cast<float4*>(x + (size_t)t * H + k) = v;
    }
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

// (sum of .x in ascending p, maximum of .y) over the nparts slice partials of token t.  Lane j
// of the (whole) warp loads partials j and j + 32, so up to 64 partials cost one round trip;
// the warp folds the shuffled values in ascending order (later partials are loaded in turn).
__device__ __forceinline__ float2 fold_partials(const float2* __restrict__ part, int t, int nparts) {
  const int lane = threadIdx.x & 31;
  const float2* pr = part + (size_t)t * nparts;
  const float2 z = make_float2(0.0f, 0.0f);
  const float2 p0 = lane < nparts ? __ldcg(pr + lane) : z;
  const float2 p1 = lane + 32 < nparts ? __ldcg(pr + lane + 32) : z;
  float ss = 0.0f, mx = 0.0f;
  const int n0 = min(nparts, 64);
  for (int p = 0; p < n0; ++p) {
    const float2 v = p < 32 ? p0 : p1;
    ss = ss + __shfl_sync(0xffffffffu, v.x, p & 31);
    mx = fmaxf(mx, __shfl_sync(0xffffffffu, v.y, p & 31));
  }
  for (int p = 64; p < nparts; ++p) {
    const float2 v = __ldcg(pr + p);
    ss = ss + v.x;
    mx = fmaxf(mx, v.y);
  }
  return make_float2(ss, mx);
}

// int8 codes of the quad (inputs k..k+3 of token t) into the activation records.  Called by a
// whole warp: lanes 8m..8m+7 hold the 32 inputs of one group (their sum seeds the group).
__device__ __forceinline__ void quant_quad(float4 v, float s, bool active, bool pad, int t, int k, uint8_t* act,
                                           int NT) {
  uint32_t codes = 0;
  int sum = 0;
  if (active) {
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
  float s, r = 1.0f;
  const float2 f = fold_partials(part, t, nparts);  // whole warps (128 threads)
  if (MODE == 1) {
    r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(f.x, (float)K), eps)));
    s = __fdiv_rn(f.y * r, 127.0f);
  } else {
    s = __fdiv_rn(f.y, 127.0f);  // the exact maximum of the partial maxima
  }
  const int k = sl * kQuantSlice + 4 * threadIdx.x;
  const bool active = k < K;  // K % 32 == 0: groups of 8 lanes are all active or all idle
  const bool pad = !active && k < chunks_of(K) * 64;  // the zero group that completes the last chunk
  float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (active) {
    v = *reinterpret_cast<const float4*>(x + (size_t)t * ldx + k);
    if (MODE == 1) { v.x = v.x * r; v.y = v.y * r; v.z = v.z * r; v.w = v.w * r; }
  }
  quant_quad(v, s, active, pad, t, k, act, act_tiles(M));
  if (sl == 0 && threadIdx.x == 0) a_s[t] = s;
}

// ------------------------------------------------------------------------- RoPE + KV

// grid (node, head among Hq query + Hkv key + Hkv value heads), D/2 threads
// The projection's output rows come from its EPI_PARTIAL slices (folded here).
// chain != 0 (a prefill bucket): token i sits at position committed_len + i.
__global__ void k_rope_kv(const SpecCtl* ctl, const TreeState* __restrict__ tree, int chain,
                          const float* __restrict__ qkv_part, int qkv_S, const float* __restrict__ a_s, int Hq, int Hkv,
                          int D, const float2* __restrict__ rope, float* kc, float* vc, int kv_cap,
                          float* __restrict__ qrot, float qscale) {
  griddep_enter();
  if (stopped(ctl)) return;
  const int i = blockIdx.x, h = blockIdx.y, j = threadIdx.x;
  const int L = (int)ctl->committed_len;
  const int pos = L + (chain ? i : tree->depth[i]);
  const int slot = L + i;
  const int half = D / 2;
  const int rows = (Hq + 2 * Hkv) * D;
  const float2 ab = mm_fold2(qkv_part, qkv_S, rows, i, h * D + j, h * D + j + half, a_s);
  const float a = ab.x, b = ab.y;
  if (h >= Hq + Hkv) {  // value head: plain copy into the cache
    float* vr = vc + ((size_t)(h - Hq - Hkv) * kv_cap + slot) * D;
    vr[j] = a;
    vr[j + half] = b;
    return;
  }
  const float2 c = rope[(size_t)pos * half + j];
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

// Merge of the split partials for wide trees: grid (node, query head), one thread per
// dimension; the same order and operations as the in-kernel merge of k_attn.
__global__ void k_attn_merge(const SpecCtl* ctl, const TreeState* __restrict__ tree, const float* __restrict__ o_part,
                             const float2* __restrict__ ml_part, int Hq, int D, int R, int splits,
                             float* __restrict__ out, float2* __restrict__ mpart) {
  griddep_enter();
  if (stopped(ctl)) return;
  __shared__ float s_mx[4];
  // row it = node i of sub-chain sub (prefill buckets hold several chains of kMaxWidth nodes)
  const int it = blockIdx.x, h = blockIdx.y, dd = threadIdx.x;
  const int sub = it / kMaxWidth, i = it - sub * kMaxWidth;
  o_part += (size_t)sub * kMaxWidth * splits * Hq * D;
  ml_part += (size_t)sub * kMaxWidth * splits * Hq;
  const int L = (int)ctl->committed_len + sub * kMaxWidth;
  const int smax = ((L + tree->depth[i]) / kAttnChunk) / R;
  const size_t hb = (size_t)i * Hq + h;
  const size_t ho = (size_t)it * Hq + h;
  const size_t sstride = (size_t)kMaxWidth * Hq;
  // the partials of splits sb .. sb + MB - 1; the maximum is taken over the first batch as it
  // arrives and over the later splits' own loads, so up to MB splits cost one round trip
  constexpr int MB = 16;
  float2 ml[MB];
  float ov[MB];
  auto load_batch = [&](int sb) {
#pragma unroll
    for (int k = 0; k < MB; ++k) {
      if (sb + k > smax) break;
      ml[k] = ml_part[(sb + k) * sstride + hb];
      ov[k] = o_part[((sb + k) * sstride + hb) * D + dd];
    }
  };
  load_batch(0);
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < MB; ++k)
    if (k <= smax) M = fmaxf(M, ml[k].x);
  for (int s2 = MB; s2 <= smax; ++s2) M = fmaxf(M, ml_part[s2 * sstride + hb].x);
  float Ls = 0.0f, O = 0.0f;
  for (int sb = 0; sb <= smax; sb += MB) {
    if (sb > 0) load_batch(sb);
#pragma unroll
    for (int k = 0; k < MB; ++k) {
      if (sb + k > smax) break;
      const float w = expf(ml[k].x - M);
      Ls = fmaf(w, ml[k].y, Ls);
      O = fmaf(w, ov[k], O);
    }
  }
  const float res = __fdiv_rn(O, Ls);
  out[ho * D + dd] = res;
  const float mx = warp_max(fabsf(res));
  if ((dd & 31) == 0) s_mx[dd >> 5] = mx;
  __syncthreads();
  if (dd == 0) {
    float m = s_mx[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, s_mx[w]);
    mpart[ho] = make_float2(0.0f, m);
  }
}

// ------------------------------------------------------------------------ SwiGLU

// grid (token, slice of kQuantSlice), 128 threads: h = silu(gate) * up written over the gate
// half of the gate|up buffer, and the slice maximum of |h|.
// gate and up rows come from the projection's EPI_PARTIAL slices (folded here).
__global__ void __launch_bounds__(kQuantSlice / 4)
    k_swiglu(const SpecCtl* ctl, const float* __restrict__ gu_part, int gu_S, const float* __restrict__ a_s,
                         float* __restrict__ gu, int F, float2* __restrict__ part) {
  griddep_enter();
  if (stopped(ctl)) return;
  __shared__ float s_mx[4];
  const int t = blockIdx.x, sl = blockIdx.y;
  const int k = sl * kQuantSlice + 4 * threadIdx.x;
  float mx = 0.0f;
  if (k < F) {
    float* g = gu + (size_t)t * 2 * F + k;
    const float4 gv = mm_fold4(gu_part, gu_S, 2 * F, t, k, a_s);
    const float4 uv = mm_fold4(gu_part, gu_S, 2 * F, t, F + k, a_s);
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
__global__ void __launch_bounds__(512)
    k_argmax(const SpecCtl* ctl, const float* __restrict__ lpart, int lS, const float* __restrict__ a_s,
                         float* __restrict__ logits, int V, float2* __restrict__ part, unsigned* __restrict__ tickets,
                         int32_t* __restrict__ pred) {
  griddep_enter();
  if (stopped(ctl)) return;
  __shared__ float sv[32];
  __shared__ int si[32];
  __shared__ unsigned s_ticket;
  const int t = blockIdx.x, sl = blockIdx.y, ns = gridDim.y;
  float* lr = logits != nullptr ? logits + (size_t)t * V : nullptr;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  const int k1 = min(V, (sl + 1) * kArgmaxSlice);
  // the head projection's slices are folded here (V % 4 == 0); the logits are stored only for
  // a caller that asked for them
  for (int k = sl * kArgmaxSlice + 4 * threadIdx.x; k < k1; k += 4 * blockDim.x) {
    const float4 v = mm_fold4(lpart, lS, V, t, k, a_s);
    if (lr != nullptr) *reinterpret_cast<float4*>(lr + k) = v;
    if (v.x > bv) { bv = v.x; bi = k; }
    if (v.y > bv) { bv = v.y; bi = k + 1; }
    if (v.z > bv) { bv = v.z; bi = k + 2; }
    if (v.w > bv) { bv = v.w; bi = k + 3; }
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

// ------------------------------------------------------------------------- code trace

// The int8 codes held by the activation records of M tokens over K inputs (the input of the
// next matmul), one thread per (token, input), written to out[t][K].  A record holds each code
// a as the f16 a, or a/16 for the inputs 8..15 and 24..31 of a group (layout.cuh).
__global__ void k_trace_codes(const uint8_t* __restrict__ act, int M, int K, int8_t* __restrict__ out) {
  griddep_enter();
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= M * K) return;
  const int t = idx / K, k = idx - t * K;
  const int NT = act_tiles(M);
  const int g = k >> 5, kin = k & 31, p = kin >> 3, tig = (kin & 7) >> 1, h = kin & 1;
  const int nt = t >> 3, gid = t & 7;
  const uint8_t* frag = act + (size_t)(g >> 1) * act_rec_bytes(NT) + (nt * 2 + (g & 1)) * 512;
  const uint32_t w = reinterpret_cast<const uint32_t*>(frag + (gid * 4 + tig) * 16)[p];
  const unsigned short bits = (unsigned short)(h ? (w >> 16) : (w & 0xffffu));
  float a = __half2float(__ushort_as_half(bits));
  if (p & 1) a *= 16.0f;
  out[(size_t)t * K + k] = (int8_t)__float2int_rn(a);
}

cudaError_t launch_trace_codes(const DecoderBufs& b, int M, int K, int8_t* out, cudaStream_t st) {
  const int n = M * K;
  return launch_pdl(k_trace_codes, dim3((n + 255) / 256), dim3(256), 0, st, (const uint8_t*)b.act, M, K, out);
}

// ------------------------------------------------------------------------- launchers

size_t attn_smem_bytes(int D, int Nq) { return attn_layout(D, Nq).total; }

namespace {
cudaError_t attn_any(int D, int G, bool configure, size_t smem, const DecoderBufs& b, const ModelDims& m, int N,
                     int layer, cudaStream_t st) {
  if (D == 64) return attn_dispatch_d64(G, configure, smem, b, m, N, layer, st);
  if (D == 128) return attn_dispatch_d128(G, configure, smem, b, m, N, layer, st);
  return cudaErrorInvalidValue;
}
}  // namespace

cudaError_t attn_tensor_maps(DecoderBufs& b, const ModelDims& m) {
  using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess) return e;
  if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorNotSupported;
  const Encode encode = reinterpret_cast<Encode>(fn);
  const cuuint64_t dims[4] = {(cuuint64_t)m.D, (cuuint64_t)b.kv_cap, (cuuint64_t)m.Hkv, (cuuint64_t)m.n_layers};
  const cuuint64_t strides[3] = {(cuuint64_t)m.D * 4, (cuuint64_t)b.kv_cap * m.D * 4,
                                 (cuuint64_t)m.Hkv * b.kv_cap * m.D * 4};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  for (int kv = 0; kv < 2; ++kv) {
    const cuuint32_t box[4] = {(cuuint32_t)(kv ? attn_vstr(m.D) : attn_kstr(m.D)), (cuuint32_t)kAttnChunk, 1, 1};
    const CUresult r = encode(kv ? &b.tm_v : &b.tm_k, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, kv ? b.vcache : b.kcache,
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

cudaError_t attn_configure(const ModelDims& m, size_t smem) {
  DecoderBufs b{};
  return attn_any(m.D, m.Hq / m.Hkv, true, smem, b, m, 1, 0, nullptr);
}

cudaError_t launch_embed(const DecoderBufs& b, const ModelDims& m, int N, bool chain, const uint32_t* ew,
                         const uint16_t* es, cudaStream_t st) {
  return launch_pdl(k_embed, dim3(N, (m.H / 8 + 127) / 128), dim3(128), 0, st, b.ctl, (const TreeState*)b.tree,
                    chain ? (const int32_t*)b.ctx : nullptr, N, ew, es, m.H, m.V, b.kv_cap, b.x);
}

cudaError_t launch_rmsnorm_quant(const DecoderBufs& b, const ModelDims& m, int N, const float* res, int res_S,
                                 cudaStream_t st) {
  const int ns = (m.H + kQuantSlice - 1) / kQuantSlice;
  cudaError_t e = launch_pdl(k_row_stats, dim3(N, ns), dim3(kQuantSlice / 4), 0, st, (const SpecCtl*)b.ctl, b.x, m.H,
                             b.qpart, res, res_S, (const float*)b.a_s);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_quant_slices<1>, dim3(N, ns), dim3(kQuantSlice / 4), 0, st, (const SpecCtl*)b.ctl,
                    (const float*)b.x, m.H, m.H, (const float2*)b.qpart, ns, m.eps, b.act, N, b.a_s);
}

cudaError_t launch_rope_kv(const DecoderBufs& b, const ModelDims& m, int N, bool chain, int layer, int qkv_S,
                           cudaStream_t st) {
  const size_t lstride = (size_t)m.Hkv * b.kv_cap * m.D;
  const float qscale = (float)(1.0 / sqrt((double)m.D));
  return launch_pdl(k_rope_kv, dim3(N, m.Hq + 2 * m.Hkv), dim3(m.D / 2), 0, st, (const SpecCtl*)b.ctl,
                    (const TreeState*)b.tree, chain ? 1 : 0, (const float*)b.mm_part, qkv_S, (const float*)b.a_s, m.Hq,
                    m.Hkv, m.D,
                    (const float2*)b.rope, b.kcache + layer * lstride,
                    b.vcache + layer * lstride, b.kv_cap, b.qrot, qscale);
}

cudaError_t launch_attention(const DecoderBufs& b, const ModelDims& m, int N, int layer, cudaStream_t st) {
  const int G = m.Hq / m.Hkv;
  const int Nn = N > kMaxWidth ? kMaxWidth : N;  // a prefill bucket runs as chains of kMaxWidth nodes
  cudaError_t e = attn_any(m.D, G, false, attn_smem_bytes(m.D, Nn * G), b, m, N, layer, st);
  if (e != cudaSuccess) return e;
  // the attention output (in the qkv buffer, [N][Hq*D]) -> int8 fragments of the O projection
  const int QD = m.Hq * m.D;
  return launch_pdl(k_quant_slices<0>, dim3(N, (QD + kQuantSlice - 1) / kQuantSlice), dim3(kQuantSlice / 4), 0, st,
                    (const SpecCtl*)b.ctl, (const float*)b.qkv, QD, QD, (const float2*)b.qpart, m.Hq, 0.0f, b.act, N,
                    b.a_s);
}

cudaError_t launch_tree_attention(const DecoderBufs& b, const ModelDims& m, int N, int layer, cudaStream_t st) {
  const int G = m.Hq / m.Hkv;
  return attn_any(m.D, G, false, attn_smem_bytes(m.D, N * G), b, m, N, layer, st);
}

cudaError_t launch_swiglu_quant(const DecoderBufs& b, const ModelDims& m, int N, int gu_S, cudaStream_t st) {
  const int ns = (m.F + kQuantSlice - 1) / kQuantSlice;
  cudaError_t e = launch_pdl(k_swiglu, dim3(N, ns), dim3(kQuantSlice / 4), 0, st, (const SpecCtl*)b.ctl,
                             (const float*)b.mm_part, gu_S, (const float*)b.a_s, b.gu, m.F, b.qpart);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_quant_slices<0>, dim3(N, ns), dim3(kQuantSlice / 4), 0, st, (const SpecCtl*)b.ctl,
                    (const float*)b.gu, m.F, 2 * m.F, (const float2*)b.qpart, ns, 0.0f, b.act, N, b.a_s);
}

cudaError_t launch_argmax(const DecoderBufs& b, const ModelDims& m, int N, int lm_S, float* logits,
                          cudaStream_t st) {
  return launch_pdl(k_argmax, dim3(N, (m.V + kArgmaxSlice - 1) / kArgmaxSlice), dim3(512), 0, st,
                    (const SpecCtl*)b.ctl, (const float*)b.mm_part, lm_S, (const float*)b.a_s, logits, m.V,
                    b.argmax_part, b.argmax_tickets, b.pred);
}

}  // namespace w4a8
