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
 * (device, both 16-byte aligned), y fp32 [M][N] (device, overwritten).  1 <= M <= 16, K % 32 == 0,
 * N % 16 == 0.  workspace: device scratch of w4a8_matmul_workspace_bytes() bytes,
 * 256-byte aligned, owned by the caller, not shared by concurrent calls; its content
 * needs no initialisation (except for w4a8_matmul_check, below).  A bounded wait inside the
 * kernel that expires makes the kernel skip its output and set the workspace status word.
 * ---------------------------------------------------------------------------- */
w4a8_status w4a8_matmul_workspace_bytes(int M, int K, int N, size_t* bytes);
w4a8_status w4a8_matmul(const int8_t* a_q, const float* a_s, int M, int K, const uint32_t* w_t,
                        const uint16_t* s_t, int N, float* y, void* workspace, size_t workspace_bytes,
                        void* stream);

/* Device.  w4a8_matmul with per-32 activation scales [P1 Small-Batch Verification Kernels:
 * activations carry one scale per block of 32 values]: a_s is fp32 [M][K/32] (device; e.g. from
 * w4a8_quantize_rows mode 1), and
 *   y[t][n] = sum_g (s_w[n][g] * s_a[t][g]) * isum[t][n][g]
 * in the fixed order of w4a8_matmul with acc = fmaf(s_w * s_a[t][g] (rounded once), isum, acc)
 * per group and no final multiply.  Same limits and workspace as w4a8_matmul. */
w4a8_status w4a8_matmul_per32(const int8_t* a_q, const float* a_s, int M, int K, const uint32_t* w_t,
                              const uint16_t* s_t, int N, float* y, void* workspace, size_t workspace_bytes,
                              void* stream);

/* Device.  The fast, non-deterministic variant of w4a8_matmul [P1 Implementation: the
 * deterministic mode fixes the reduction order at a cost the paper measures as 0-15%]: the same
 * exact integer group sums and per-slice fmaf chains, but the K slices of each output are added
 * into y (zeroed by this call) with float atomics in arrival order instead of the fixed left fold,
 * so the last bits of y may vary between calls and M tokens need not give the bits of M single
 * calls.  Same arguments, limits and workspace as w4a8_matmul (the workspace status word reports
 * an expired wait; the split-K partial area is not used). */
w4a8_status w4a8_matmul_nondet(const int8_t* a_q, const float* a_s, int M, int K, const uint32_t* w_t,
                               const uint16_t* s_t, int N, float* y, void* workspace, size_t workspace_bytes,
                               void* stream);

/* Host, synchronous.  Reads the device status word of a matmul workspace (call after the
 * stream has finished).  *flags = 0 if every bounded pipeline wait of the kernels that
 * used this workspace completed; otherwise it holds W4A8_FLAG_ERR_TIMEOUT (16) and the call
 * returns W4A8_ERR_DEVICE_FLAG.  The workspace must be zero-filled once before its first use for
 * this word to be meaningful. */
w4a8_status w4a8_matmul_check(const void* workspace, int M, int K, int N, uint32_t* flags);

/* Device, test-only fault injection without a fault [P2 "WebGPU for LLM Inference, in depth":
 * error scopes and device loss -- a failed submission is reported, the device stays usable].
 * Same arguments as w4a8_matmul; the matmul kernel runs in a variant whose copy warp issues no
 * copy, so every consumer's bounded wait (shortened to 1 ms) expires: the kernel sets the
 * workspace status word to W4A8_FLAG_ERR_TIMEOUT (read it with w4a8_matmul_check), leaves y
 * unwritten, has no copy in flight and returns.  Nothing hangs or faults; later calls on the
 * same device work normally.  The production kernels are separate instantiations. */
w4a8_status w4a8_matmul_inject_timeout(const int8_t* a_q, const float* a_s, int M, int K, const uint32_t* w_t,
                                       const uint16_t* s_t, int N, float* y, void* workspace, size_t workspace_bytes,
                                       void* stream);

/* Device.  The same product as w4a8_matmul (same kernels, same bits) for callers that
 * cannot allocate device memory -- e.g. code already inside a CUDA stream capture, or hosts
 * that give the library only its inputs and outputs.  It allocates nothing: its scratch is a
 * 32 MiB array in the library's device image (held by every GPU that loads the library until
 * the process exits); shapes whose scratch would exceed it return W4A8_ERR_CAPACITY before
 * any launch.  The array's device address is looked up on the first call on each device, so
 * that first call should come before any stream capture.  All calls share the array and it
 * keeps the last call's contents (each call clears what must start at zero): calls that can
 * overlap on the GPU (different streams, or threads without ordering) race and must not be
 * issued.  A bounded wait inside the kernel that expires leaves y incomplete and sets the
 * array's status word, which w4a8_matmul_noalloc_check reads.  The paper has no counterpart of
 * this entry point. */
w4a8_status w4a8_matmul_noalloc(const int8_t* a_q, const float* a_s, int M, int K, const uint32_t* w_t,
                                const uint16_t* s_t, int N, float* y, void* stream);

/* Host, synchronous.  The status word of the last w4a8_matmul_noalloc call on the current
 * device (call after that call's stream has finished; a later call clears it): *flags = 0 if
 * every bounded pipeline wait of its kernels completed, else W4A8_FLAG_ERR_TIMEOUT (16), y was
 * left incomplete and the call returns W4A8_ERR_DEVICE_FLAG.  Allocates nothing.  The paper has
 * no counterpart of this entry point. */
w4a8_status w4a8_matmul_noalloc_check(uint32_t* flags);

/* Number of K slices S that w4a8_matmul uses for a (K, N) shape (host). */
int w4a8_matmul_slices(int K, int N);

/* ==============================================================================
 * Decoder, session and the GPU-resident speculation loop
 * ============================================================================ */

/* Shape of a Llama/Qwen-style decoder without biases, RMSNorm gain 1, rotate-half RoPE
 * [P1 Experiments (models); Implementation].  hidden % 32 == 0, ffn % 32 == 0,
 * (n_heads + 2 n_kv_heads) * head_dim % 16 == 0, head_dim in {64, 128},
 * n_heads % n_kv_heads == 0, n_heads / n_kv_heads <= 8 (<= 4 at head_dim 128: the tree
 * attention of 16 nodes holds all query heads of a KV head in one CTA's shared memory),
 * vocab % 16 == 0; else W4A8_ERR_SHAPE. */
typedef struct {
  int n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab;
  int tied;         /* 1: the LM head is the embedding table */
  float rms_eps;    /* RMSNorm epsilon */
  float rope_base;  /* RoPE base (theta_i = base^(-2i/head_dim)) */
} w4a8_model_desc;

/* Tensor kinds for w4a8_model_load_tensor; [rows][cols] of each (P2 layout, device):
 *   Q [n_heads*head_dim][hidden], K and V [n_kv_heads*head_dim][hidden],
 *   O [hidden][n_heads*head_dim], GATE and UP [ffn][hidden], DOWN [hidden][ffn],
 *   EMBED and LM_HEAD [vocab][hidden] (LM_HEAD only when not tied). */
enum {
  W4A8_T_Q = 0, W4A8_T_K = 1, W4A8_T_V = 2, W4A8_T_O = 3, W4A8_T_GATE = 4, W4A8_T_UP = 5, W4A8_T_DOWN = 6,
  W4A8_T_EMBED = 7, W4A8_T_LM_HEAD = 8
};

typedef struct w4a8_model w4a8_model;
typedef struct w4a8_session w4a8_session;

/* Host.  Allocates the model's device weight storage (tiled layout, fused QKV and
 * GATE|UP matrices).  The weights must then be loaded with w4a8_model_load_tensor. */
w4a8_status w4a8_model_create(const w4a8_model_desc* desc, w4a8_model** out);
/* Device.  Copies one quantised tensor (P2 layout, device, caller-owned; may be freed
 * after the stream has passed this call) into the model.  layer is ignored for EMBED and
 * LM_HEAD. */
w4a8_status w4a8_model_load_tensor(w4a8_model* m, int kind, int layer, const uint32_t* w_p2,
                                   const uint16_t* s_p2, void* stream);
/* Host.  Device bytes held by the model's weights. */
w4a8_status w4a8_model_weight_bytes(const w4a8_model* m, size_t* bytes);
void w4a8_model_destroy(w4a8_model* m);

typedef struct {
  int kv_cap;       /* KV slots per layer (>= prompt + max_new + max_width) */
  int ctx_cap;      /* context token capacity (>= prompt + max_new + 9) */
  int max_window;   /* largest window W of spec_window (1..64) */
  int eos_id;       /* stop token, or -1 */
  int mem_cap;      /* session-memory entries (0..32768; ctx_cap + mem_cap <= 225280), 0 = none */
} w4a8_session_desc;

/* The 32-byte device control state [P1 GPU-Resident Speculation Loop]. */
typedef struct {
  uint32_t committed_len;  /* KV entries committed (all context tokens except the root) */
  uint32_t ctx_len;        /* context tokens (prompt + generated); the last one is the root */
  uint32_t n_valid;        /* valid nodes of the current full-width draft tree */
  int32_t root_tok;        /* node 0 of the next step */
  uint32_t n_generated;    /* tokens generated since the prompt */
  uint32_t max_new;        /* generation stops at this many tokens */
  uint32_t flags;          /* W4A8_FLAG_* */
  uint32_t step_idx;       /* steps executed */
} w4a8_ctl;

/* The 16-byte host summary of the control state read between windows. */
typedef struct {
  uint32_t committed_len, n_generated, flags;
  int32_t root_tok;
} w4a8_ctl16;

#define W4A8_FLAG_TERMINATED 1u     /* max_new reached or eos emitted */
#define W4A8_FLAG_ERR_CAPACITY 2u   /* kv_cap or ctx_cap would be exceeded */
#define W4A8_FLAG_ERR_TOKEN 4u      /* a token id outside [0, vocab) */
#define W4A8_FLAG_ERR_TREE 8u       /* malformed tree */
#define W4A8_FLAG_ERR_TIMEOUT 16u   /* a bounded device wait expired */

/* Per-step statistics written by accept_greedy, 12 bytes [P1 GPU-Resident Speculation
 * Loop; Feedback Control]: accepted draft nodes, match length of the drafter's best
 * candidate, valid tree nodes, tokens emitted, low 32 bits of the device timer (ns) at
 * the end of acceptance. */
typedef struct {
  uint16_t n_accepted_drafts, best_match_len, n_nodes, n_emitted;
  uint32_t t_lo;
} w4a8_step_stats;

/* Host.  Allocates a session's device state (KV cache fp32 [layers][kv heads][kv_cap]
 * [head_dim], context, control, activations, scratch) and pinned host mirrors. */
w4a8_status w4a8_session_create(w4a8_model* m, const w4a8_session_desc* desc, w4a8_session** out);
void w4a8_session_destroy(w4a8_session* s);

/* Device.  Starts a generation: context = prompt[0..n) (device int32), KV of
 * prompt[0..n-1) computed through the verification kernels in buckets of 64 tokens (the
 * matmuls and row-wise kernels take a whole bucket, the attention four chains of 16), the
 * rest as one pass over its whole chains of 16 and one shorter chain
 * ("GPU-Resident Speculative Decoding ...", Design >
 * Small-Batch Verification Kernels: token buckets), root = prompt[n-1], n_generated = 0,
 * then the first draft tree.  The cache holds the bits of sequential single-token steps. */
w4a8_status w4a8_prefill(w4a8_session* s, const int32_t* prompt, int n, int max_new, void* stream);

/* Device.  One verification pass over tree nodes 0..N-1 [P1 GPU-Resident Speculation
 * Loop]: node i at logical position committed_len + depth(i) writes its K/V to slot
 * committed_len + i and attends to cache slots [0, committed_len) and to its ancestors;
 * pred[i] = argmax of its logits (lowest index on ties).  logits: optional device
 * fp32 [N][vocab] copy of the logits (NULL = none).  1 <= N <= 16. */
w4a8_status tree_verify_step(w4a8_session* s, int N, float* logits, void* stream);
/* Host.  Bytes of the code trace of a verification pass of N tokens (1 <= N <= 16):
 * N * (n_layers * (2 * hidden + n_heads * head_dim + ffn) + hidden). */
w4a8_status w4a8_model_trace_bytes(const w4a8_model* m, int N, size_t* bytes);
/* Device.  tree_verify_step that also writes the int8 activation codes the matmuls consumed
 * [P1 Small-Batch Verification Kernels: int8 activations quantised right before each matrix
 * multiplication], for tests and tools: codes (device int8, codes_bytes >= the size from
 * w4a8_model_trace_bytes) receives, for each layer in order, the codes of the RMSNorm output
 * before Q/K/V [N][hidden], of the attention output before O [N][n_heads*head_dim], of the
 * RMSNorm output before gate/up [N][hidden] and of the SwiGLU output before down [N][ffn],
 * then those of the final RMSNorm output before the LM head [N][hidden].  W4A8_ERR_CAPACITY if
 * the buffer is too small (nothing is launched). */
w4a8_status w4a8_tree_verify_trace(w4a8_session* s, int N, float* logits, int8_t* codes, size_t codes_bytes,
                                   void* stream);
/* Device.  Greedy acceptance [P1; P3 section 4]: walks from the root following the
 * lowest-index child whose token equals its parent's prediction; commits the accepted
 * drafts and the bonus token (at most max_new - n_generated, stopping after eos); updates
 * the control state, the context and the statistics. */
w4a8_status accept_greedy(w4a8_session* s, int N, void* stream);
/* Device.  Moves the accepted path's K/V rows to consecutive slots [P1; P3 section 7]. */
w4a8_status kv_compact(w4a8_session* s, void* stream);
/* Device.  Suffix n-gram drafter [P1 Draft-Free Drafting]: next tree of 16 nodes in
 * best-first order (its first N nodes are the tree of width N). */
w4a8_status ngram_draft(w4a8_session* s, void* stream);
/* Device.  tree_verify_step + accept_greedy + kv_compact + ngram_draft. */
w4a8_status w4a8_spec_step(w4a8_session* s, int N, void* stream);

/* Device.  Launches W speculation steps of width N as one CUDA graph (captured on first
 * use per (N, W)), followed by an asynchronous copy of the control state, the W step
 * statistics and the emitted tokens into pinned host memory [P1 GPU-Resident Speculation
 * Loop: windows of W steps, two windows in flight].  At most two windows may be in
 * flight; the first call for a new (N, W) must not happen during stream capture. */
w4a8_status spec_window(w4a8_session* s, int N, int W, void* stream);
/* Host.  Waits (at most timeout_us microseconds; < 0 = no limit) for the oldest window in
 * flight and returns its results: control summary, step statistics (*n_stats <= W) and
 * emitted tokens (*n_tokens; tokens must hold 16 * W entries).  W4A8_ERR_TIMEOUT leaves the
 * window in flight; W4A8_ERR_ARG if no window is in flight. */
w4a8_status spec_poll(w4a8_session* s, w4a8_ctl16* ctl, w4a8_step_stats* stats, int* n_stats,
                      int32_t* tokens, int* n_tokens, int64_t timeout_us);

/* Host, synchronous.  Device-timed cost T(N) of one verification step plus drafting for
 * each width [P1 Feedback Control: measured at load time], median of `trials` trials of
 * `reps` back-to-back graph launches each; the session state is left unchanged. */
w4a8_status w4a8_calibrate(w4a8_session* s, const int* widths, int n_widths, int reps, int trials,
                           float* t_us);

typedef struct {
  int max_new;          /* tokens to generate */
  int window;           /* W, steps per graph launch (1..max_window) */
  int fixed_width;      /* > 0: every step uses this width; 0: the width controller */
  int in_flight;        /* windows in flight (1 or 2) */
  int64_t timeout_us;   /* per-window wait limit (< 0: none) */
  int n_widths;         /* controller widths (ascending) and their costs T(N) in us */
  int widths[8];
  float t_us[8];
} w4a8_decode_opts;

typedef struct {
  int n_tokens, n_steps, n_windows, host_syncs;
  int accepted_drafts;  /* sum over steps */
  int width_steps[17];  /* steps per width */
  uint32_t flags;       /* final control flags */
  double device_us;     /* device time from the first to the last step end */
  int64_t kernels;      /* kernel launches of the windows run (kernel nodes of their graphs) */
} w4a8_decode_report;

/* Host, synchronous: the end-to-end call.  prompt: host int32[n_prompt]; out: host
 * int32[max_new].  Copies the prompt to the device, prefills, then runs windows of
 * speculation steps with `in_flight` windows in flight, choosing each window's width
 * with the width controller (or fixed_width) between windows. */
w4a8_status w4a8_decode(w4a8_session* s, const int32_t* prompt, int n_prompt, const w4a8_decode_opts* opts,
                        int32_t* out, int* n_out, w4a8_decode_report* report, void* stream);

/* Device.  ORs W4A8_FLAG_* bits into the control word between kernels: TERMINATED cancels
 * the generation; an error bit makes every later kernel of the session a no-op (the host
 * sees it in the next window's control summary).  Used for cancellation and for
 * host-side fault injection in tests. */
w4a8_status w4a8_session_raise_flags(w4a8_session* s, uint32_t flags, void* stream);

/* Host, synchronous: the window loop of w4a8_decode on a session already prefilled by
 * w4a8_prefill (the prompt and the KV cache stay resident on the device).  out: host
 * int32[max_new of the prefill]; opts->max_new is ignored (the prefill fixed it). */
w4a8_status w4a8_generate(w4a8_session* s, const w4a8_decode_opts* opts, int32_t* out, int* n_out,
                          w4a8_decode_report* report, void* stream);

/* Host, synchronous.  Device time of the matmul launches of one verification pass of
 * width N (every layer and the LM head, nothing else) captured in one CUDA graph and
 * replayed `reps` times: average microseconds per launch and average algorithmic bytes
 * per launch (packed weights + scales + int8 activations + fp32 outputs). */
w4a8_status w4a8_time_matmuls(w4a8_session* s, int N, int reps, double* us_per_launch, double* bytes_per_launch,
                              int* launches_per_pass);

/* Host, synchronous state access (tests and tools). */
w4a8_status w4a8_session_get_ctl(w4a8_session* s, w4a8_ctl* ctl);
/* Replaces the current tree: tok/parent host int32[n] with parent[0] = -1 and
 * 0 <= parent[i] < i; nodes n..15 become padding. */
w4a8_status w4a8_session_set_tree(w4a8_session* s, const int32_t* tok, const int32_t* parent, int n);
w4a8_status w4a8_session_get_tree(w4a8_session* s, int32_t* tok, int32_t* parent, int32_t* depth, int* n_valid,
                                  int* best_len);
w4a8_status w4a8_session_get_pred(w4a8_session* s, int32_t* pred, int n);
/* Copies the context tokens (host int32[cap]); *n = context length. */
w4a8_status w4a8_session_get_context(w4a8_session* s, int32_t* out, int cap, int* n);
/* Session memory [P1 Draft-Free Drafting From Web Context: the drafter's scan also covers a
 * buffer of the model's outputs from earlier requests; Experiments: a 32K-token budget].  The
 * memory holds earlier outputs, each preceded by the separator -1, oldest first, in at most
 * mem_cap entries (whole outputs are dropped from the oldest; an output longer than the memory
 * keeps its last mem_cap - 1 tokens).  The drafter scans it as if it preceded the context: a
 * match or a continuation never crosses a separator, and among equal match lengths a context
 * position counts as more recent than any memory position.  It enters neither the KV cache nor
 * the prefill.  Host, synchronous; not while windows are in flight (W4A8_ERR_ARG).
 * append: tokens host int32[n] in [0, vocab); W4A8_ERR_CAPACITY if the session has mem_cap < 2.
 * get: copies min(cap, entries) entries to out (host) and sets *n to the number of entries. */
w4a8_status w4a8_session_memory_append(w4a8_session* s, const int32_t* tokens, int n);
w4a8_status w4a8_session_memory_clear(w4a8_session* s);
w4a8_status w4a8_session_memory_get(const w4a8_session* s, int32_t* out, int cap, int* n);

/* Tree attention of one layer alone [P1 GPU-Resident Speculation Loop: each node attends to
 * the committed cache and to its ancestors], on the session's cache, committed length L and tree,
 * for caller-supplied queries: node i (0 <= i < n) attends to cache slots [0, L) and to the
 * slots L + a of its ancestors-or-self a, with softmax weights over q . k.
 * q: device fp32 [n][n_heads][head_dim], queries after RoPE and the 1/sqrt(head_dim) scale
 * (query head h uses KV head h / (n_heads / n_kv_heads)); out: device fp32
 * [n][n_heads * head_dim].  Slots L .. L+n-1 must hold the nodes' K/V (tree_verify_step
 * writes them).  Synchronises the stream to read the control state: W4A8_ERR_DEVICE_FLAG
 * if a stop or error flag is set, W4A8_ERR_CAPACITY if L + n > kv_cap, W4A8_ERR_ARG if
 * n exceeds the tree's valid nodes.  Overwrites the session's query and attention
 * scratch buffers (tests and tools). */
w4a8_status w4a8_session_attention(w4a8_session* s, int layer, int n, const float* q, float* out, void* stream);
/* Device.  The inverse of w4a8_session_copy_kv: writes K and V of one layer, slots
 * [slot0, slot0+n), from k_in/v_in (device fp32 [n_kv_heads][n][head_dim]) into the cache, e.g.
 * to restore a saved cache or to verify on a given cache [P1 GPU-Resident Speculation Loop: the
 * committed KV cache is the state a verification step reads].  The control state is unchanged. */
w4a8_status w4a8_session_load_kv(w4a8_session* s, int layer, int slot0, int n, const float* k_in, const float* v_in,
                                 void* stream);
/* Device.  Copies K and V of one layer, slots [slot0, slot0+n), into k_out/v_out (device
 * fp32 [n_kv_heads][n][head_dim]). */
w4a8_status w4a8_session_copy_kv(w4a8_session* s, int layer, int slot0, int n, float* k_out, float* v_out,
                                 void* stream);

/* ------------------------------------------------------------------------------
 * Width controller [P1 Feedback Control of Speculation Width], host only.
 * Chooses N maximising E[tokens per step | N] / T(N), where E is estimated from the
 * recent best match lengths and the acceptance observed per (width, match length);
 * probes a wider tree after a run of width-1 windows (spacing set by the costs, doubled
 * up to 64 windows after each probe window that accepts no draft, reset by one that does;
 * windows must be observed in the order they were chosen);
 * refines T(N) with an exponential moving average of the device-measured window
 * completion intervals.
 * ---------------------------------------------------------------------------- */
typedef struct w4a8_controller w4a8_controller;
w4a8_status w4a8_controller_create(const int* widths, const float* t_us, int n, w4a8_controller** out);
void w4a8_controller_destroy(w4a8_controller* c);
/* Width for the next window. */
int w4a8_controller_choose(w4a8_controller* c);
/* Feeds one finished window: its width, its step statistics and the device interval
 * (us) since the previous window's end (<= 0: unknown). */
w4a8_status w4a8_controller_observe(w4a8_controller* c, int width, const w4a8_step_stats* stats, int n,
                                    double interval_us);
/* Expected tokens per step of a width at the current statistics (for tests/reports). */
double w4a8_controller_expected_tokens(const w4a8_controller* c, int width);
/* Current cost estimate T(N) in us. */
double w4a8_controller_cost(const w4a8_controller* c, int width);

#ifdef __cplusplus
}
#endif

#endif /* W4A8_H */
