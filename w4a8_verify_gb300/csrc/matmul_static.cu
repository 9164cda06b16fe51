// w4a8_matmul without any allocation: the scratch (activation records, split-K partials,
// slice counters and a status word) lives in one file-scope device array instead of a
// caller-provided workspace.
//
// Why: some callers of this library cannot call cudaMalloc -- code that is already inside a
// CUDA stream capture (an allocation is not a stream operation), hosts that hand the
// library only the input and output buffers, or latency-critical paths that must not pay
// for an allocation's implicit synchronisation.  They still own and pass inputs and outputs.
#include <mutex>

#include "matmul.cuh"

using namespace w4a8;

namespace {

// Upper bound of the scratch of one call; every GPU that loads this library holds it
// until the process exits.
constexpr size_t kStaticScratchBytes = (size_t)32 << 20;

__device__ __align__(256) unsigned char g_mm_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

inline size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Device address of g_mm_scratch on the current device (looked up once per device; the
// host-side name is only a stand-in for the device array and must not be passed to kernels).
w4a8_status scratch_address(void** out) {
  int dev = 0;
  W4A8_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return W4A8_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    W4A8_CUDA_TRY(cudaGetSymbolAddress(&p, g_mm_scratch));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return W4A8_OK;
}

}  // namespace

W4A8_API w4a8_status w4a8_matmul_noalloc(const int8_t* a_q, const float* a_s, int M, int K, const uint32_t* w_t,
                                         const uint16_t* s_t, int N, float* y, void* stream) {
  if (!a_q || !a_s || !w_t || !s_t || !y || M <= 0 || K <= 0 || N <= 0) return W4A8_ERR_ARG;
  if (M > 16 || K % 32 || N % 16) return W4A8_ERR_SHAPE;
  if (!aligned(w_t, 16) || !aligned(s_t, 16) || !aligned(a_q, 4) || !aligned(a_s, 4)) return W4A8_ERR_ARG;
  const MatmulPlan p = mm_plan(K, N);
  // [status word, n_rg slice counters][activation records][split-K partials]: the status word
  // sits at offset 0 for every shape, so that w4a8_matmul_noalloc_check can find it
  const size_t off_act = align256(((size_t)p.n_rg + 1) * 4);
  const size_t off_part = align256(off_act + act_bytes(K));
  const size_t total = off_part + p.part_floats * 4;
  if (total > kStaticScratchBytes) return W4A8_ERR_CAPACITY;
  void* base_v = nullptr;
  const w4a8_status st = scratch_address(&base_v);
  if (st != W4A8_OK) return st;
  char* base = static_cast<char*>(base_v);
  unsigned* status = reinterpret_cast<unsigned*>(base);
  uint8_t* act = reinterpret_cast<uint8_t*>(base + off_act);
  float* part = reinterpret_cast<float*>(base + off_part);
  cudaStream_t cs = as_stream(stream);
  // the fragment pass also zeroes the status word and the slice counters that follow it: the
  // array keeps the previous call's contents, and these must start at zero
  W4A8_CUDA_TRY(act_prep_run(a_q, M, K, K, act, status, p.n_rg + 1, cs));
  W4A8_CUDA_TRY(mm_run(p, w_t, s_t, act, a_s, M, y, N, EPI_STORE, part, status + 1, status, nullptr, cs));
  return W4A8_OK;
}

W4A8_API w4a8_status w4a8_matmul_noalloc_check(uint32_t* flags) {
  if (!flags) return W4A8_ERR_ARG;
  void* base = nullptr;
  const w4a8_status st = scratch_address(&base);
  if (st != W4A8_OK) return st;
  W4A8_CUDA_TRY(cudaMemcpy(flags, base, 4, cudaMemcpyDeviceToHost));
  return *flags ? W4A8_ERR_DEVICE_FLAG : W4A8_OK;
}
