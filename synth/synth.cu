// Device side of the counter-based input generator of synth/gen.py (same definitions,
// bit for bit).  Input generation only: no arithmetic of the decoding method.
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#define SYNTH_API extern "C" __attribute__((visibility("default")))

namespace {
constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t fin(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
__device__ __forceinline__ uint64_t sm64(uint64_t k, uint64_t i) { return fin(k + (i + 1) * kGolden); }

__device__ __forceinline__ float normal_at(uint64_t key, uint64_t e, float mult) {
  int64_t s = 0;
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const uint64_t w = sm64(key, 3 * e + j);
#pragma unroll
    for (int b = 0; b < 4; ++b) s += (int64_t)((w >> (16 * b)) & 0xFFFFull);
  }
  return __fmul_rn((float)(s - 393210), mult);
}

__global__ void k_normal(uint64_t key, uint64_t start, uint64_t count, float mult, float* out) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < count; i += (uint64_t)gridDim.x * blockDim.x)
    out[i] = normal_at(key, start + i, mult);
}

// rows [row0, row0+nrows) of a [rows][cols] tensor whose real extent is real_rows x real_cols
__global__ void k_dense(uint64_t key, int cols, int real_rows, int real_cols, long long row0, long long nrows,
                        float mult, float* out) {
  const uint64_t total = (uint64_t)nrows * cols;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < total; i += (uint64_t)gridDim.x * blockDim.x) {
    const long long r = row0 + (long long)(i / cols);
    const int c = (int)(i % cols);
    float v = 0.0f;
    if (r < real_rows && c < real_cols) v = normal_at(key, (uint64_t)r * real_cols + c, mult);
    out[i] = v;
  }
}

__global__ void k_codes(uint64_t key, uint64_t start, uint64_t count, int8_t* out) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < count; i += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t e = start + i;
    const uint64_t w = sm64(key, e / 16);
    out[i] = (int8_t)((int)((w >> (4 * (e % 16))) & 15ull) - 8);
  }
}

__global__ void k_scales(uint64_t key, uint64_t start, uint64_t count, float range, float lo, uint16_t* out) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < count; i += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t w = sm64(key, start + i);
    const float u = __fmul_rn((float)(w >> 40), 5.9604644775390625e-08f);  // 2^-24
    const float v = __fadd_rn(__fmul_rn(u, range), lo);
    out[i] = __half_as_ushort(__float2half_rn(v));
  }
}

inline int blocks_for(uint64_t n) {
  uint64_t b = (n + 255) / 256;
  return (int)(b > 65536 ? 65536 : (b == 0 ? 1 : b));
}
}  // namespace

SYNTH_API int synth_normal(uint64_t key, uint64_t start, uint64_t count, float mult, float* out, void* stream) {
  k_normal<<<blocks_for(count), 256, 0, (cudaStream_t)stream>>>(key, start, count, mult, out);
  return (int)cudaGetLastError();
}
SYNTH_API int synth_dense(uint64_t key, int cols, int real_rows, int real_cols, long long row0, long long nrows,
                          float mult, float* out, void* stream) {
  k_dense<<<blocks_for((uint64_t)nrows * cols), 256, 0, (cudaStream_t)stream>>>(key, cols, real_rows, real_cols, row0,
                                                                                nrows, mult, out);
  return (int)cudaGetLastError();
}
SYNTH_API int synth_codes(uint64_t key, uint64_t start, uint64_t count, int8_t* out, void* stream) {
  k_codes<<<blocks_for(count), 256, 0, (cudaStream_t)stream>>>(key, start, count, out);
  return (int)cudaGetLastError();
}
SYNTH_API int synth_scales(uint64_t key, uint64_t start, uint64_t count, float range, float lo, uint16_t* out,
                           void* stream) {
  k_scales<<<blocks_for(count), 256, 0, (cudaStream_t)stream>>>(key, start, count, range, lo, out);
  return (int)cudaGetLastError();
}
