// Tree attention kernels of head size 64 (one translation unit per head size, compiled in
// parallel).
#include "attention.cuh"

namespace w4a8 {

cudaError_t attn_dispatch_d64(int G, bool configure, size_t smem, const DecoderBufs& b, const ModelDims& m, int N,
                              int layer, cudaStream_t st) {
  return attn_dispatch_g<64>(G, configure, smem, b, m, N, layer, st);
}

}  // namespace w4a8
