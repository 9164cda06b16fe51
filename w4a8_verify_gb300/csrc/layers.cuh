// Launchers of the decoder kernels (layers.cu) and the speculation kernels (spec.cu).
#pragma once
#include "decoder.cuh"

namespace w4a8 {

size_t attn_smem_bytes(int D, int Nq);
cudaError_t attn_configure(const ModelDims& m, size_t smem);
// encodes b.tm_k and b.tm_v (the caches must be allocated)
cudaError_t attn_tensor_maps(DecoderBufs& b, const ModelDims& m);

// chain: a prefill bucket (tokens committed_len + i of the context at positions committed_len + i);
// otherwise the current tree's nodes
cudaError_t launch_embed(const DecoderBufs& b, const ModelDims& m, int N, bool chain, const uint32_t* ew,
                         const uint16_t* es, cudaStream_t st);
// res: EPI_PARTIAL slices (res_S of them) of the projection whose output is added to the
// residual stream x before the statistics, or nullptr
cudaError_t launch_rmsnorm_quant(const DecoderBufs& b, const ModelDims& m, int N, const float* res, int res_S,
                                 cudaStream_t st);
// the QKV projection's output comes from its qkv_S EPI_PARTIAL slices in b.mm_part
cudaError_t launch_rope_kv(const DecoderBufs& b, const ModelDims& m, int N, bool chain, int layer, int qkv_S,
                           cudaStream_t st);
// N > kMaxWidth (a prefill bucket, a multiple of kMaxWidth): N / kMaxWidth chains of kMaxWidth nodes
// (the current tree must be the chain of kMaxWidth nodes)
cudaError_t launch_attention(const DecoderBufs& b, const ModelDims& m, int N, int layer, cudaStream_t st);
// the tree attention pass alone: queries b.qrot -> attention output in b.qkv ([N][Hq*D])
cudaError_t launch_tree_attention(const DecoderBufs& b, const ModelDims& m, int N, int layer, cudaStream_t st);
// gate|up from the gu_S EPI_PARTIAL slices in b.mm_part
cudaError_t launch_swiglu_quant(const DecoderBufs& b, const ModelDims& m, int N, int gu_S, cudaStream_t st);
// logits from the lm_S EPI_PARTIAL slices of the head projection in b.mm_part (folded here and
// stored to `logits` [N][vocab] when it is not null)
cudaError_t launch_argmax(const DecoderBufs& b, const ModelDims& m, int N, int lm_S, float* logits, cudaStream_t st);

// int8 codes of the current activation records (M tokens, K inputs) -> out [M][K]
cudaError_t launch_trace_codes(const DecoderBufs& b, int M, int K, int8_t* out, cudaStream_t st);

// spec.cu
cudaError_t launch_accept(const DecoderBufs& b, int N, int window_slot, cudaStream_t st);
cudaError_t launch_compact(const DecoderBufs& b, const ModelDims& m, cudaStream_t st);
cudaError_t launch_draft(const DecoderBufs& b, int force, cudaStream_t st);
// scan_cap: context plus session-memory capacity (bytes of the drafter's shared scan array)
cudaError_t draft_configure(int scan_cap);
cudaError_t launch_chain_tree(const DecoderBufs& b, int start, int len, cudaStream_t st);
cudaError_t launch_commit_chain(const DecoderBufs& b, int len, cudaStream_t st);

}  // namespace w4a8
