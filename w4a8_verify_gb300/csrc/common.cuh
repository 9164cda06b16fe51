// Shared helpers of the sm_103a kernels: status handling, launch with programmatic
// dependent launch, warp reductions, e4m3 encoding of small integers.
#pragma once
#include <cstdint>
#include <cstddef>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include "../../include/w4a8.h"

#define W4A8_API extern "C" __attribute__((visibility("default")))

#define W4A8_CUDA_TRY(expr)                                  \
  do {                                                       \
    cudaError_t _e = (expr);                                 \
    if (_e != cudaSuccess) {                                 \
      (void)cudaGetLastError();                              \
      return W4A8_ERR_CUDA;                                  \
    }                                                        \
  } while (0)

namespace w4a8 {

// Device error / state flags (the session control word and the matmul status word).
enum : uint32_t {
  FLAG_TERMINATED = 1u,
  FLAG_ERR_CAPACITY = 2u,
  FLAG_ERR_TOKEN = 4u,
  FLAG_ERR_TREE = 8u,
  FLAG_ERR_TIMEOUT = 16u,
  FLAG_ERR_MASK = FLAG_ERR_CAPACITY | FLAG_ERR_TOKEN | FLAG_ERR_TREE | FLAG_ERR_TIMEOUT,
  FLAG_STOP_MASK = FLAG_TERMINATED | FLAG_ERR_MASK,
};

static inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Launch with the programmatic-stream-serialization attribute: the kernel may start
// while its predecessor drains; it must execute griddep_wait() before touching any
// memory the predecessor writes or reads.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// e4m3 byte of a small integer (|v| <= 128 and exactly representable); exact.
__device__ __forceinline__ uint32_t e4m3_of_int(int v) {
  return (uint32_t)__nv_cvt_float_to_fp8((float)v, __NV_SATFINITE, __NV_E4M3);
}

// Split of an int8 activation a = 16*hi + lo, hi in [-8,7], lo in [0,15]; returns the
// e4m3 bytes of 16*hi and of lo (both exact).
__device__ __forceinline__ void split_act(int a, uint32_t& hi_byte, uint32_t& lo_byte) {
  int hi = a >> 4;  // arithmetic shift: floor(a / 16)
  int lo = a & 15;
  hi_byte = e4m3_of_int(16 * hi);
  lo_byte = e4m3_of_int(lo);
}

}  // namespace w4a8
