// Device state of a decoding session and the launchers of the decoder kernels.
//
// "GPU-Resident Speculative Decoding ..." (Design > GPU-Resident Speculation Loop):
// the state a CPU would normally keep -- committed KV length, number of valid nodes,
// context length, termination flag -- lives in a small device buffer that every kernel
// reads at run time, so a whole window of steps needs no host decision.
#pragma once
#include "matmul.cuh"

namespace w4a8 {

constexpr int kMaxWidth = 16;     // tree nodes per step (node 0 = last committed token)
constexpr int kMaxBucket = 64;    // prompt tokens per prefill bucket (four chains of kMaxWidth for attention)
constexpr int kMaxCont = 8;       // drafter continuation length -> at most 9 tokens per step
constexpr int kAttnChunk = 64;    // logical positions per attention chunk (fixed: part of the order)

// 32-byte control state (device).
struct SpecCtl {
  uint32_t committed_len;  // L_c: KV slots holding committed tokens (all context tokens but the root)
  uint32_t ctx_len;        // tokens in the context buffer (prompt + generated); last one is the root
  uint32_t n_valid;        // valid nodes of the current tree (drafted at full width)
  int32_t root_tok;        // node 0 of the next step = last context token
  uint32_t n_generated;    // tokens emitted since the prompt
  uint32_t max_new;        // stop after this many generated tokens
  uint32_t flags;          // FLAG_*
  uint32_t step_idx;       // steps executed
};
static_assert(sizeof(SpecCtl) == 32, "control state is 32 bytes");

// Current draft tree (full width; a step of width N uses nodes 0..N-1, a prefix-closed set).
struct TreeState {
  int32_t tok[kMaxWidth];
  int32_t parent[kMaxWidth];  // parent[0] = -1, parent[i] < i
  int32_t depth[kMaxWidth];
  int32_t n_valid;            // nodes >= n_valid are padding (token 0, child of the root)
  int32_t best_len;           // match length of the drafter's best candidate
  int32_t pad[2];
};

// What accept_greedy did in the last step, for kv_compact.
struct AcceptRec {
  int32_t valid;     // 1 if the last accept committed tokens
  int32_t L_old;     // committed_len before the step
  int32_t n_commit;  // KV entries committed (= tokens emitted)
  int32_t n_path;    // accepted path length including the root
  int32_t path[kMaxWidth];
};

// Per-step statistics (12 bytes), written by accept_greedy.
struct StepStats {
  uint16_t n_accepted_drafts;
  uint16_t best_match_len;
  uint16_t n_nodes;
  uint16_t n_emitted;
  uint32_t t_lo;  // low 32 bits of %globaltimer (ns) at the end of acceptance
};
static_assert(sizeof(StepStats) == 12, "stats are 12 bytes");

struct ModelDims {
  int n_layers, H, Hq, Hkv, D, F, V, tied;
  float eps, rope_base;
  int qkv_rows() const { return (Hq + 2 * Hkv) * D; }
};

// Device buffers the decoder kernels use (pointers into a session's allocation).
struct DecoderBufs {
  SpecCtl* ctl;
  TreeState* tree;
  AcceptRec* rec;
  int32_t* ctx;
  int32_t* pred;          // [16]
  float* x;               // [kMaxBucket][H] residual stream
  float* qkv;             // [kMaxBucket][qkv_rows] (the attention output [kMaxBucket][Hq*D] too)
  float* qrot;            // [kMaxBucket][Hq][D]
  float* gu;              // [kMaxBucket][2F]
  float* o_part;          // attention split partials [chain][split][16][Hq][D] (split < n_chunks, 2 chains)
  float* ml_part;         // [chain][split][16][Hq] (running max, sum)
  uint8_t* act;           // activation records of the next matmul (max K)
  float* a_s;             // [kMaxBucket] activation scales
  float* mm_part;         // split-K partials
  unsigned* tickets;      // split-K counters (zero between kernels)
  float* kcache;          // [L][Hkv][kv_cap][D]
  float* vcache;
  float2* rope;           // [kv_cap][D/2] (cos, sin)
  float2* qpart;          // [kMaxBucket][slices] (sum of squares, max |x|) partials of the quantisation passes
  float2* argmax_part;    // [16][vocab slices] (value, index) partials
  unsigned* argmax_tickets;  // [16], zero between kernels
  unsigned* attn_tickets;    // [2 chains][Hkv], zero between kernels
  int32_t* mem;           // [mem_cap] session memory: earlier outputs, each preceded by -1
  int* mem_len;           // entries of mem in use (device word, read by the drafter)
  StepStats* wstats;      // [max_window] current window's statistics
  int32_t* wtok;          // [max_window][16] emitted tokens per step of the window
  int kv_cap, ctx_cap, n_chunks, max_window, mem_cap;
  int eos_id;
  // TMA maps of the K and V caches, dims {D, kv_cap, Hkv, layers}; a box is one attention
  // chunk of 64 rows landing at the padded shared-memory row strides
  CUtensorMap tm_k, tm_v;
};

}  // namespace w4a8
