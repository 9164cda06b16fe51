// Shared helpers of the sm_103a kernels: status handling, launch with programmatic
// dependent launch, warp reductions, e4m3 encoding of small integers.
#pragma once
#include <cstdint>
#include <cstddef>
#include <cuda.h>
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
// Kernel entry: wait for the preceding grid, then let the next kernel of the stream be
// scheduled at once; its CTAs block in their own griddepcontrol.wait until this grid has
// completed and its writes are visible, so only the launch latency overlaps.
__device__ __forceinline__ void griddep_enter() {
  griddep_wait();
  griddep_launch();
}

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

// ---- mbarrier / bulk-copy helpers (CTA scope) ----------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: gives up after kWaitLimitNs and reports false.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (unsigned it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
  }
}
// TMA tiled copy of one 4-D box (coordinates innermost first) of `map` into shared memory;
// its bytes complete on bar.  x must keep the box start 16-byte aligned.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace w4a8
