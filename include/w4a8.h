/*
 * w4a8.h -- C ABI of the GB300 (sm_103a) library for GPU-resident tree-speculative
 * greedy decoding with W4A8 small-batch verification.
 *
 * Sources (cited by page title and section):
 *   [P1] "GPU-Resident Speculative Decoding for In-Browser LLM Inference with WebGPU":
 *        Design > Small-Batch Verification Kernels; Design > GPU-Resident Speculation
 *        Loop; Design > Draft-Free Drafting From Web Context; Design > Feedback Control
 *        of Speculation Width; Implementation.
 *   [P2] "WebGPU for LLM Inference, in depth": section "A quantised matrix-vector
 *        kernel in WGSL" (packed int4 layout).
 *   [P3] "Exact Speculative And Assisted Decoding For A Tiny Draft And Qualified
 *        Champion": section 4 (greedy acceptance, bonus token), section 7 (KV commit
 *        and rollback as a logical-length move).
 *
 * Conventions shared by every entry point:
 *   - Every function returns a w4a8_status (0 = success) and never aborts or prints.
 *   - Pointers documented "device" must point to device memory of the current CUDA
 *     device; "host" pointers to host memory.  The caller owns every buffer it
 *     passes; the library never frees caller memory.  Opaque handles own only the
 *     memory they allocate and release it in their destroy function.
 *   - Work is asynchronous on the given stream (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream) unless the comment says "synchronous".
 *   - fp16 values cross the ABI as uint16_t bit patterns.
 *   - Argument errors are detected on the host before any launch (status
 *     W4A8_ERR_ARG / W4A8_ERR_SHAPE); CUDA launch failures return W4A8_ERR_CUDA.
 */
#ifndef W4A8_H
#define W4A8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  W4A8_OK = 0,
  W4A8_ERR_ARG = 1,          /* null pointer or out-of-range scalar argument */
  W4A8_ERR_SHAPE = 2,        /* a dimension breaks a layout rule (e.g. K % 32 != 0) */
  W4A8_ERR_UNSUPPORTED = 3,  /* valid request the library does not implement */
  W4A8_ERR_CAPACITY = 4,     /* KV / context / workspace capacity exceeded */
  W4A8_ERR_CUDA = 5,         /* a CUDA runtime call failed */
  W4A8_ERR_TIMEOUT = 6,      /* a bounded host wait expired */
  W4A8_ERR_DEVICE_FLAG = 7,  /* a kernel reported an error through the control flags */
  W4A8_ERR_NOMEM = 8         /* device or pinned host allocation failed */
} w4a8_status;

/* Text for a status code (static storage). */
const char* w4a8_status_str(int status);

/* Version of this ABI (incremented on incompatible changes). */
int w4a8_abi_version(void);

/* ------------------------------------------------------------------------------
 * Weight format
 *
 * [P1 Small-Batch Verification Kernels] weights are 4-bit codes with one 16-bit
 * scale per 32 inputs; [P2 quantised matvec] eight codes per u32, code j of word k
 * is element 8k+j in bits 4j..4j+3, stored as 0..15 meaning -8..7.
 *
 * "P2 layout" of a [N][K] weight (K % 32 == 0):
 *   words  u32 [N][K/8]   (row-major)
 *   scales fp16 [N][K/32]
 * "Tiled layout" (this library's internal layout for the tensor-core matmul, made by
 * w4a8_repack_weights; sizes from w4a8_weight_layout_bytes): 16-row blocks x 64-input
 * chunks so that one warp load feeds one mma.sync fragment.
 * ---------------------------------------------------------------------------- */

/* Host, synchronous.  Packs int8 codes q[N][K] (values in [-8,7]) into P2 words
 * w_out[N][K/8].  K % 8 == 0.  Returns W4A8_ERR_ARG if a code is out of range. */
w4a8_status w4a8_pack_weights(const int8_t* q, int N, int K, uint32_t* w_out);

/* Device.  Offline converter [P1 Implementation]: symmetric int4 quantisation of a
 * fp32 weight w[N][K] (device) in groups of 32 along K:
 *   s = fp16(fp32(absmax) / 7),  q = clamp(rint(w / s), -8, 7)  (fp32, round half even),
 *   absmax == 0 or s == 0 -> s = 0, q = 0.
 * Writes P2 words w_p2[N][K/8] and scales s_p2[N][K/32] (device).  K % 32 == 0. */
w4a8_status w4a8_quantize_weights(const float* w, int N, int K, uint32_t* w_p2, uint16_t* s_p2,
                                  void* stream);

/* Host.  Bytes of the tiled layout of a [N][K] weight (N % 16 == 0, K % 32 == 0). */
w4a8_status w4a8_weight_layout_bytes(int N, int K, size_t* words_bytes, size_t* scales_bytes);

/* Device.  P2 layout (w_p2, s_p2) -> tiled layout (w_t, s_t).  N % 16 == 0, K % 32 == 0.
 * If K % 64 == 32 the tiled layout ends with one zero group (code 0, scale 0). */
w4a8_status w4a8_repack_weights(const uint32_t* w_p2, const uint16_t* s_p2, int N, int K,
                                uint32_t* w_t, uint16_t* s_t, void* stream);

/* ------------------------------------------------------------------------------
 * Activation quantisation [P1 Small-Batch Verification Kernels]: int8 codes with a
 * fp32 scale, mode 0 = one scale per token row (absmax of the row), mode 1 = one
 * scale per block of 32 values.  Rule (fp32, IEEE division, round half even):
 *   s = absmax / 127,  q = clamp(rint(x / s), -127, 127);  absmax == 0 -> s = 0, q = 0.
 * x[M][K] fp32 (device) -> q[M][K] int8, s[M] (mode 0) or s[M][K/32] (mode 1) (device).
 * ---------------------------------------------------------------------------- */
w4a8_status w4a8_quantize_rows(const float* x, int M, int K, int mode, int8_t* q, float* s,
                               void* stream);

/* ------------------------------------------------------------------------------
 * W4A8 small-batch matmul [P1 Small-Batch Verification Kernels; Implementation:
 * deterministic mode]:
 *   y[t][n] = s_a[t] * sum_g s_w[n][g] * isum[t][n][g],
 *   isum[t][n][g] = sum_{k in group g} q_w[n][k] * q_a[t][k]   (exact integer)
 * Fixed fp32 order (independent of M, so M tokens give the bits of M single calls):
 * the groups are split into S contiguous slices (S a function of K and N only); in a
 * slice acc = fmaf(s_w, isum, acc) over ascending groups from 0; the slice results
 * are folded left in ascending slice order; y = fold * s_a[t].
 *
 * a_q int8 [M][K], a_s fp32 [M] (device; per-token mode), w_t/s_t tiled layout
 * (device), y fp32 [M][N] (device, overwritten).  1 <= M <= 16, K % 32 == 0,
 * N % 16 == 0.  workspace: device scratch of w4a8_matmul_workspace_bytes() bytes,
 * 256-byte aligned, owned by the caller, not shared by concurrent calls; its content
 * needs no initialisation.
 * ---------------------------------------------------------------------------- */
w4a8_status w4a8_matmul_workspace_bytes(int M, int K, int N, size_t* bytes);
w4a8_status w4a8_matmul(const int8_t* a_q, const float* a_s, int M, int K, const uint32_t* w_t,
                        const uint16_t* s_t, int N, float* y, void* workspace, size_t workspace_bytes,
                        void* stream);

/* Number of K slices S that w4a8_matmul uses for a (K, N) shape (host). */
int w4a8_matmul_slices(int K, int N);

#ifdef __cplusplus
}
#endif

#endif /* W4A8_H */
