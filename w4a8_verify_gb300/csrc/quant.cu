// Weight and activation quantisation, the packed int4 layouts and their conversion.
//
// "GPU-Resident Speculative Decoding ..." (Design > Small-Batch Verification Kernels;
// Implementation): 4-bit weight codes with one 16-bit scale per 32 inputs, int8
// activations.  "WebGPU for LLM Inference, in depth" (quantised matvec in WGSL): eight
// codes per u32, code j of word k = element 8k+j, stored 0..15 meaning -8..7.
#include "common.cuh"
#include "layout.cuh"

using namespace w4a8;

W4A8_API const char* w4a8_status_str(int s) {
  switch (s) {
    case W4A8_OK: return "ok";
    case W4A8_ERR_ARG: return "invalid argument";
    case W4A8_ERR_SHAPE: return "unsupported shape";
    case W4A8_ERR_UNSUPPORTED: return "unsupported request";
    case W4A8_ERR_CAPACITY: return "capacity exceeded";
    case W4A8_ERR_CUDA: return "CUDA error";
    case W4A8_ERR_TIMEOUT: return "timeout";
    case W4A8_ERR_DEVICE_FLAG: return "device error flag";
    case W4A8_ERR_NOMEM: return "out of memory";
    default: return "unknown status";
  }
}

W4A8_API int w4a8_abi_version(void) { return 2; }

W4A8_API w4a8_status w4a8_pack_weights(const int8_t* q, int N, int K, uint32_t* w_out) {
  if (!q || !w_out || N <= 0 || K <= 0) return W4A8_ERR_ARG;
  if (K % 8) return W4A8_ERR_SHAPE;
  const size_t words = (size_t)K / 8;
  for (size_t r = 0; r < (size_t)N; ++r) {
    for (size_t w = 0; w < words; ++w) {
      uint32_t acc = 0;
      for (int j = 0; j < 8; ++j) {
        int v = q[r * (size_t)K + w * 8 + j];
        if (v < -8 || v > 7) return W4A8_ERR_ARG;
        acc |= (uint32_t)(v + 8) << (4 * j);
      }
      w_out[r * words + w] = acc;
    }
  }
  return W4A8_OK;
}

// One warp per (row, group of 32): absmax (exact), fp16 scale, codes, 4 packed words.
__global__ void k_quantize_weights(const float* __restrict__ w, int N, int K, uint32_t* __restrict__ wq,
                                   uint16_t* __restrict__ ws) {
  griddep_enter();
  const int G = K / 32;
  const long long item = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (item >= (long long)N * G) return;
  const int lane = threadIdx.x & 31;
  const long long row = item / G;
  const int g = (int)(item % G);
  const float v = w[row * K + (long long)g * 32 + lane];
  const float amax = warp_max(fabsf(v));
  const __half s16 = __float2half_rn(__fdiv_rn(amax, 7.0f));
  const float s32 = __half2float(s16);
  int q = 0;
  if (s32 > 0.0f) {
    float r = rintf(__fdiv_rn(v, s32));
    r = fminf(fmaxf(r, -8.0f), 7.0f);
    q = (int)r;
  }
  uint32_t nib = (uint32_t)(q + 8) << (4 * (lane & 7));
  // OR the 8 nibbles of each word (lanes 8j..8j+7)
  nib |= __shfl_xor_sync(0xffffffffu, nib, 1);
  nib |= __shfl_xor_sync(0xffffffffu, nib, 2);
  nib |= __shfl_xor_sync(0xffffffffu, nib, 4);
  if ((lane & 7) == 0) wq[row * (K / 8) + (long long)g * 4 + lane / 8] = nib;
  if (lane == 0) ws[row * G + g] = (s32 > 0.0f) ? __half_as_ushort(s16) : (uint16_t)0;
}

W4A8_API w4a8_status w4a8_quantize_weights(const float* w, int N, int K, uint32_t* w_p2, uint16_t* s_p2,
                                           void* stream) {
  if (!w || !w_p2 || !s_p2 || N <= 0 || K <= 0) return W4A8_ERR_ARG;
  if (K % 32) return W4A8_ERR_SHAPE;
  const long long items = (long long)N * (K / 32);
  const int warps = 8;
  const long long blocks = (items + warps - 1) / warps;
  if (blocks > 0x7fffffffLL) return W4A8_ERR_SHAPE;
  W4A8_CUDA_TRY(launch_pdl(k_quantize_weights, dim3((unsigned)blocks), dim3(32 * warps), 0, as_stream(stream),
                           w, N, K, w_p2, s_p2));
  return W4A8_OK;
}

W4A8_API w4a8_status w4a8_weight_layout_bytes(int N, int K, size_t* words_bytes, size_t* scales_bytes) {
  if (N <= 0 || K <= 0 || !words_bytes || !scales_bytes) return W4A8_ERR_ARG;
  if (N % 16 || K % 32) return W4A8_ERR_SHAPE;
  *words_bytes = tiled_words(N, K) * 4;
  *scales_bytes = tiled_scales(N, K) * 2;
  return W4A8_OK;
}

// One thread per output word of the tiled layout (see layout.cuh).  The source rows
// [0, N) land at rows [row0, row0 + N) of an Ntot-row tiled matrix.
__global__ void k_repack_words(const uint32_t* __restrict__ wp2, int N, int K, int Ntot, int row0,
                               uint32_t* __restrict__ wt) {
  griddep_enter();
  const long long total = (long long)tiled_words(N, K);
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int KC = chunks_of(K);
  const int G = K / 32;
  const int j = (int)(i & 3);
  const int lane = (int)((i >> 2) & 31);
  const long long rc = i >> 7;  // source (rb, c)
  const int c = (int)(rc % KC);
  const int rb = (int)(rc / KC);
  const int gid = lane >> 2, tig = lane & 3;
  const long long row = (long long)rb * 16 + gid + ((j & 1) ? 8 : 0);
  const int g = 2 * c + (j >> 1);
  uint32_t out = 0x88888888u;  // code 0 in every nibble for a padding group
  if (g < G) {
    out = 0;
    const uint32_t* src = wp2 + row * (K / 8);
    for (int p = 0; p < 4; ++p)
      for (int h = 0; h < 2; ++h) {
        const int k = 32 * g + 8 * p + 2 * tig + h;
        const uint32_t n = (src[k >> 3] >> (4 * (k & 7))) & 15u;
        out |= n << (4 * p + 16 * h);
      }
  }
  const size_t t = tile_index(Ntot, KC, row0 / 16 + rb, c);
  wt[t * 128 + (i & 127)] = out;
}

__global__ void k_repack_scales(const uint16_t* __restrict__ sp2, int N, int K, int Ntot, int row0,
                                uint16_t* __restrict__ st) {
  griddep_enter();
  const long long total = (long long)tiled_scales(N, K);
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int KC = chunks_of(K);
  const int G = K / 32;
  const int j = (int)(i & 3);
  const int gid = (int)((i >> 2) & 7);
  const long long rc = i >> 5;
  const int c = (int)(rc % KC);
  const int rb = (int)(rc / KC);
  const long long row = (long long)rb * 16 + gid + ((j & 1) ? 8 : 0);
  const int g = 2 * c + (j >> 1);
  const size_t t = tile_index(Ntot, KC, row0 / 16 + rb, c);
  st[t * 32 + (i & 31)] = (g < G) ? sp2[row * G + g] : (uint16_t)0;
}

namespace w4a8 {
cudaError_t repack_run(const uint32_t* w_p2, const uint16_t* s_p2, int N, int K, int Ntot, int row0, uint32_t* w_t,
                       uint16_t* s_t, cudaStream_t st) {
  const long long nw = (long long)tiled_words(N, K), ns = (long long)tiled_scales(N, K);
  cudaError_t e =
      launch_pdl(k_repack_words, dim3((unsigned)((nw + 255) / 256)), dim3(256), 0, st, w_p2, N, K, Ntot, row0, w_t);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_repack_scales, dim3((unsigned)((ns + 255) / 256)), dim3(256), 0, st, s_p2, N, K, Ntot, row0,
                    s_t);
}
}  // namespace w4a8

W4A8_API w4a8_status w4a8_repack_weights(const uint32_t* w_p2, const uint16_t* s_p2, int N, int K,
                                         uint32_t* w_t, uint16_t* s_t, void* stream) {
  if (!w_p2 || !s_p2 || !w_t || !s_t || N <= 0 || K <= 0) return W4A8_ERR_ARG;
  if (N % 16 || K % 32) return W4A8_ERR_SHAPE;
  if (!aligned(w_t, 16) || !aligned(s_t, 16)) return W4A8_ERR_ARG;
  const long long nw = (long long)tiled_words(N, K), ns = (long long)tiled_scales(N, K);
  if ((nw + 255) / 256 > 0x7fffffffLL) return W4A8_ERR_SHAPE;
  (void)ns;
  W4A8_CUDA_TRY(repack_run(w_p2, s_p2, N, K, N, 0, w_t, s_t, as_stream(stream)));
  return W4A8_OK;
}

// Per-token mode: one CTA (256 threads) per row.  absmax is exact in any order.
__global__ void k_quantize_rows_token(const float* __restrict__ x, int K, int8_t* __restrict__ q,
                                      float* __restrict__ s) {
  griddep_enter();
  __shared__ float red[8];
  const int row = blockIdx.x;
  const float* xr = x + (size_t)row * K;
  float m = 0.0f;
  for (int k = threadIdx.x; k < K; k += blockDim.x) m = fmaxf(m, fabsf(xr[k]));
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  float amax = red[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) amax = fmaxf(amax, red[w]);
  const float sc = __fdiv_rn(amax, 127.0f);
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    int v = 0;
    if (sc > 0.0f) v = (int)fminf(fmaxf(rintf(__fdiv_rn(xr[k], sc)), -127.0f), 127.0f);
    q[(size_t)row * K + k] = (int8_t)v;
  }
  if (threadIdx.x == 0) s[row] = sc;
}

// Per-32 mode: one warp per (row, block).
__global__ void k_quantize_rows_block(const float* __restrict__ x, int M, int K, int8_t* __restrict__ q,
                                      float* __restrict__ s) {
  griddep_enter();
  const int G = K / 32;
  const long long item = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (item >= (long long)M * G) return;
  const int lane = threadIdx.x & 31;
  const float v = x[item * 32 + lane];
  const float amax = warp_max(fabsf(v));
  const float sc = __fdiv_rn(amax, 127.0f);
  int r = 0;
  if (sc > 0.0f) r = (int)fminf(fmaxf(rintf(__fdiv_rn(v, sc)), -127.0f), 127.0f);
  q[item * 32 + lane] = (int8_t)r;
  if (lane == 0) s[item] = sc;
}

W4A8_API w4a8_status w4a8_quantize_rows(const float* x, int M, int K, int mode, int8_t* q, float* s,
                                        void* stream) {
  if (!x || !q || !s || M <= 0 || K <= 0) return W4A8_ERR_ARG;
  cudaStream_t st = as_stream(stream);
  if (mode == 0) {
    W4A8_CUDA_TRY(launch_pdl(k_quantize_rows_token, dim3(M), dim3(256), 0, st, x, K, q, s));
  } else if (mode == 1) {
    if (K % 32) return W4A8_ERR_SHAPE;
    const long long items = (long long)M * (K / 32);
    W4A8_CUDA_TRY(launch_pdl(k_quantize_rows_block, dim3((unsigned)((items + 7) / 8)), dim3(256), 0, st, x, M,
                             K, q, s));
  } else {
    return W4A8_ERR_ARG;
  }
  return W4A8_OK;
}
