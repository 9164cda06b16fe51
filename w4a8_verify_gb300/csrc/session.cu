// Host side of the decoder: model and session objects, prefill, the verification pass,
// the speculation step, CUDA-graph windows with pinned read-back, calibration and the
// end-to-end decode loop.
//
// "GPU-Resident Speculative Decoding ..." (Design > GPU-Resident Speculation Loop): no step
// needs a decision of the CPU, so a window of W steps is encoded as one submission (here one
// CUDA graph) and two windows are kept in flight; the CPU reads only the 32-byte control
// state and 12 bytes of statistics per step of the finished window, copied by the same
// submission into mapped (pinned) host memory.  (Feedback Control): step costs measured
// on the device at load time; the width is chosen between windows.
#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstring>
#include <deque>
#include <map>
#include <new>
#include <vector>

#include "decoder.cuh"
#include "layers.cuh"

using namespace w4a8;

namespace {
struct Arena {
  std::vector<void*> dev, host;
  ~Arena() {
    for (void* p : dev) cudaFree(p);
    for (void* p : host) cudaFreeHost(p);
  }
  template <class T>
  bool dalloc(T** p, size_t bytes) {
    void* q = nullptr;
    if (cudaMalloc(&q, bytes ? bytes : 256) != cudaSuccess) {
      (void)cudaGetLastError();
      return false;
    }
    dev.push_back(q);
    *p = static_cast<T*>(q);
    return true;
  }
  template <class T>
  bool halloc(T** p, size_t bytes) {
    void* q = nullptr;
    if (cudaMallocHost(&q, bytes ? bytes : 256) != cudaSuccess) {
      (void)cudaGetLastError();
      return false;
    }
    host.push_back(q);
    *p = static_cast<T*>(q);
    return true;
  }
};

#define TRYC(expr)                           \
  do {                                       \
    cudaError_t _e = (expr);                 \
    if (_e != cudaSuccess) return _e;        \
  } while (0)

constexpr int kMaxWindow = 64;
constexpr int kMaxMemory = 32768;  // session-memory entries (the pages' 32K-token budget)
constexpr int kRecBytesFixed = 32;
constexpr int kRecStepBytes = (int)sizeof(StepStats) + kMaxWidth * 4;
}  // namespace

struct w4a8_model {
  ModelDims d{};
  int qkv_rows = 0;
  Arena arena;
  uint32_t* emb_w = nullptr;  // P2 layout copy for the lookup
  uint16_t* emb_s = nullptr;
  uint32_t* lm_w = nullptr;  // tiled
  uint16_t* lm_s = nullptr;
  std::vector<uint32_t*> qkv_w, o_w, gu_w, dn_w;
  std::vector<uint16_t*> qkv_s, o_s, gu_s, dn_s;
  MatmulPlan p_qkv{}, p_o{}, p_gu{}, p_dn{}, p_lm{};
  size_t bytes = 0;
};

struct w4a8_session {
  w4a8_model* m = nullptr;
  Arena arena;
  DecoderBufs b{};
  int max_window = 1;
  uint8_t* dev_rec = nullptr;        // packed window record (device)
  uint8_t* host_rec[2] = {nullptr, nullptr};
  int32_t* pin = nullptr;            // pinned staging for host <-> device state
  int32_t* prompt_dev = nullptr;
  cudaEvent_t ev[2] = {nullptr, nullptr};
  cudaStream_t cap = nullptr;
  struct Flight {
    int slot, W, N;
  };
  std::deque<Flight> q;
  std::vector<int32_t> mem_host;           // host copy of the session memory
  int next_slot = 0;
  std::map<long long, cudaGraphExec_t> graphs;
  std::map<long long, int> graph_kernels;  // kernel nodes of each window graph
  cudaGraphExec_t bucket_graph = nullptr;  // one prefill bucket of kMaxBucket prompt tokens
  long long host_syncs = 0;
  long long kernels = 0;                   // kernels launched by window graphs
  ~w4a8_session() {
    for (auto& kv : graphs) cudaGraphExecDestroy(kv.second);
    if (bucket_graph) cudaGraphExecDestroy(bucket_graph);
    for (int i = 0; i < 2; ++i)
      if (ev[i]) cudaEventDestroy(ev[i]);
    if (cap) cudaStreamDestroy(cap);
  }
};

namespace {

inline long long graph_key(int N, int W, int slot) { return ((long long)N << 32) | ((long long)W << 8) | slot; }

__global__ void k_init_ctl(SpecCtl* ctl, AcceptRec* rec, const int32_t* ctx, int n, int max_new) {
  griddep_enter();
  if (threadIdx.x != 0) return;
  SpecCtl c;
  c.committed_len = 0;
  c.ctx_len = (uint32_t)n;
  c.n_valid = 1;
  c.root_tok = ctx[n - 1];
  c.n_generated = 0;
  c.max_new = (uint32_t)max_new;
  c.flags = max_new <= 0 ? FLAG_TERMINATED : 0u;
  c.step_idx = 0;
  *ctl = c;
  rec->valid = 0;
}

// Packs the control state, the window's step statistics and emitted tokens contiguously.
__global__ void k_window_close(const SpecCtl* ctl, const StepStats* ws, const int32_t* wt, int W, uint8_t* out) {
  griddep_enter();
  const int t = threadIdx.x;
  if (t < 8) reinterpret_cast<uint32_t*>(out)[t] = reinterpret_cast<const uint32_t*>(ctl)[t];
  StepStats* so = reinterpret_cast<StepStats*>(out + kRecBytesFixed);
  int32_t* to = reinterpret_cast<int32_t*>(out + kRecBytesFixed + (size_t)W * sizeof(StepStats));
  for (int i = t; i < W; i += blockDim.x) so[i] = ws[i];
  for (int i = t; i < W * kMaxWidth; i += blockDim.x) to[i] = wt[i];
}

// Bytes of the code trace of one verification pass of N tokens: per layer the codes of the
// four quantisation points (RMSNorm -> QKV, attention -> O, RMSNorm -> gate|up, SwiGLU -> down),
// then the final RMSNorm -> LM head, each [N][inputs].
size_t trace_bytes(const ModelDims& d, int N) {
  return (size_t)N * ((size_t)d.n_layers * (2 * d.H + d.Hq * d.D + d.F) + d.H);
}

// trace: optional device buffer of trace_bytes(d, N) bytes receiving the int8 codes of every
// quantisation point (tests and tools; not used by the decoding loop).
// chain: N (a multiple of kMaxWidth, at most kMaxBucket) context tokens from committed_len (the
// current tree must be the chain of kMaxWidth nodes, which the attention takes for each chain);
// otherwise the current tree's first N nodes.
cudaError_t forward(w4a8_session* s, int N, bool head, float* logits_out, cudaStream_t st, int8_t* trace = nullptr,
                    bool chain = false) {
  const DecoderBufs& b = s->b;
  w4a8_model* m = s->m;
  const ModelDims& d = m->d;
  unsigned* flags = &b.ctl->flags;
  TRYC(launch_embed(b, d, N, chain, m->emb_w, m->emb_s, st));
  // The layer projections leave per-slice partial sums (EPI_PARTIAL) that the next kernel
  // folds: RoPE/KV, the residual update before RMSNorm, SwiGLU.
  const float* res = nullptr;
  int res_S = 0;
  int8_t* tr = trace;
  auto trace_codes = [&](int K) -> cudaError_t {
    if (!tr) return cudaSuccess;
    cudaError_t e = launch_trace_codes(b, N, K, tr, st);
    tr += (size_t)N * K;
    return e;
  };
  for (int l = 0; l < d.n_layers; ++l) {
    TRYC(launch_rmsnorm_quant(b, d, N, res, res_S, st));
    TRYC(trace_codes(d.H));
    TRYC(mm_run(m->p_qkv, m->qkv_w[l], m->qkv_s[l], b.act, b.a_s, N, nullptr, 0, EPI_PARTIAL, b.mm_part, b.tickets,
                flags, flags, st));
    TRYC(launch_rope_kv(b, d, N, chain, l, m->p_qkv.S, st));
    TRYC(launch_attention(b, d, N, l, st));
    TRYC(trace_codes(d.Hq * d.D));
    TRYC(mm_run(m->p_o, m->o_w[l], m->o_s[l], b.act, b.a_s, N, nullptr, 0, EPI_PARTIAL, b.mm_part, b.tickets, flags,
                flags, st));
    TRYC(launch_rmsnorm_quant(b, d, N, b.mm_part, m->p_o.S, st));
    TRYC(trace_codes(d.H));
    TRYC(mm_run(m->p_gu, m->gu_w[l], m->gu_s[l], b.act, b.a_s, N, nullptr, 0, EPI_PARTIAL, b.mm_part, b.tickets,
                flags, flags, st));
    TRYC(launch_swiglu_quant(b, d, N, m->p_gu.S, st));
    TRYC(trace_codes(d.F));
    TRYC(mm_run(m->p_dn, m->dn_w[l], m->dn_s[l], b.act, b.a_s, N, nullptr, 0, EPI_PARTIAL, b.mm_part, b.tickets,
                flags, flags, st));
    res = b.mm_part;
    res_S = m->p_dn.S;
  }
  if (head) {
    TRYC(launch_rmsnorm_quant(b, d, N, res, res_S, st));
    TRYC(trace_codes(d.H));
    TRYC(mm_run(m->p_lm, m->lm_w, m->lm_s, b.act, b.a_s, N, nullptr, 0, EPI_PARTIAL, b.mm_part, b.tickets, flags,
                flags, st));
    TRYC(launch_argmax(b, d, N, m->p_lm.S, logits_out, st));
  }
  return cudaSuccess;
}

cudaError_t step(w4a8_session* s, int N, int wslot, cudaStream_t st) {
  TRYC(forward(s, N, true, nullptr, st));
  TRYC(launch_accept(s->b, N, wslot, st));
  TRYC(launch_compact(s->b, s->m->d, st));
  return launch_draft(s->b, 0, st);
}

w4a8_status sync_read(w4a8_session* s, void* host, const void* dev, size_t bytes) {
  W4A8_CUDA_TRY(cudaMemcpy(host, dev, bytes, cudaMemcpyDeviceToHost));
  return W4A8_OK;
}

}  // namespace

// ------------------------------------------------------------------------------ model

W4A8_API w4a8_status w4a8_model_create(const w4a8_model_desc* desc, w4a8_model** out) {
  if (!desc || !out) return W4A8_ERR_ARG;
  const w4a8_model_desc& d = *desc;
  if (d.n_layers <= 0 || d.hidden <= 0 || d.n_heads <= 0 || d.n_kv_heads <= 0 || d.ffn <= 0 || d.vocab <= 0)
    return W4A8_ERR_ARG;
  if (d.hidden % 32 || d.ffn % 32 || d.vocab % 16 || d.n_heads % d.n_kv_heads) return W4A8_ERR_SHAPE;
  if (d.head_dim != 64 && d.head_dim != 128) return W4A8_ERR_SHAPE;
  if (d.n_heads / d.n_kv_heads > 8) return W4A8_ERR_SHAPE;
  // the attention's dynamic shared memory for 16 nodes x all query heads of a KV head, plus
  // room for its static arrays, within one block's opt-in limit (227 KB)
  constexpr size_t kMaxSmemPerBlock = 232448, kAttnStaticRoom = 4096;
  if (attn_smem_bytes(d.head_dim, kMaxWidth * (d.n_heads / d.n_kv_heads)) + kAttnStaticRoom > kMaxSmemPerBlock)
    return W4A8_ERR_SHAPE;
  if (((d.n_heads + 2 * d.n_kv_heads) * d.head_dim) % 16) return W4A8_ERR_SHAPE;
  if (!(d.rms_eps >= 0.0f) || !(d.rope_base > 0.0f)) return W4A8_ERR_ARG;
  w4a8_model* m = new (std::nothrow) w4a8_model();
  if (!m) return W4A8_ERR_NOMEM;
  m->d = ModelDims{d.n_layers, d.hidden, d.n_heads, d.n_kv_heads, d.head_dim, d.ffn, d.vocab, d.tied ? 1 : 0,
                   d.rms_eps, d.rope_base};
  const int H = d.hidden, F = d.ffn, QD = d.n_heads * d.head_dim;
  m->qkv_rows = (d.n_heads + 2 * d.n_kv_heads) * d.head_dim;
  m->p_qkv = mm_plan(H, m->qkv_rows);
  m->p_o = mm_plan(QD, H);
  m->p_gu = mm_plan(H, 2 * F);
  m->p_dn = mm_plan(F, H);
  m->p_lm = mm_plan(H, d.vocab);
  auto tw = [](int N, int K) { return tiled_words(N, K) * 4; };
  auto ts = [](int N, int K) { return tiled_scales(N, K) * 2; };
  bool ok = true;
  m->qkv_w.resize(d.n_layers); m->qkv_s.resize(d.n_layers);
  m->o_w.resize(d.n_layers); m->o_s.resize(d.n_layers);
  m->gu_w.resize(d.n_layers); m->gu_s.resize(d.n_layers);
  m->dn_w.resize(d.n_layers); m->dn_s.resize(d.n_layers);
  for (int l = 0; l < d.n_layers && ok; ++l) {
    ok = ok && m->arena.dalloc(&m->qkv_w[l], tw(m->qkv_rows, H)) && m->arena.dalloc(&m->qkv_s[l], ts(m->qkv_rows, H));
    ok = ok && m->arena.dalloc(&m->o_w[l], tw(H, QD)) && m->arena.dalloc(&m->o_s[l], ts(H, QD));
    ok = ok && m->arena.dalloc(&m->gu_w[l], tw(2 * F, H)) && m->arena.dalloc(&m->gu_s[l], ts(2 * F, H));
    ok = ok && m->arena.dalloc(&m->dn_w[l], tw(H, F)) && m->arena.dalloc(&m->dn_s[l], ts(H, F));
    m->bytes += tw(m->qkv_rows, H) + ts(m->qkv_rows, H) + tw(H, QD) + ts(H, QD) + tw(2 * F, H) + ts(2 * F, H) +
                tw(H, F) + ts(H, F);
  }
  ok = ok && m->arena.dalloc(&m->emb_w, (size_t)d.vocab * H / 2) && m->arena.dalloc(&m->emb_s, (size_t)d.vocab * H / 16);
  ok = ok && m->arena.dalloc(&m->lm_w, tw(d.vocab, H)) && m->arena.dalloc(&m->lm_s, ts(d.vocab, H));
  m->bytes += (size_t)d.vocab * H / 2 + (size_t)d.vocab * H / 16 + tw(d.vocab, H) + ts(d.vocab, H);
  if (!ok) {
    delete m;
    return W4A8_ERR_NOMEM;
  }
  *out = m;
  return W4A8_OK;
}

W4A8_API w4a8_status w4a8_model_load_tensor(w4a8_model* m, int kind, int layer, const uint32_t* w_p2,
                                            const uint16_t* s_p2, void* stream) {
  if (!m || !w_p2 || !s_p2) return W4A8_ERR_ARG;
  const ModelDims& d = m->d;
  const int H = d.H, F = d.F, QD = d.Hq * d.D, KVD = d.Hkv * d.D;
  cudaStream_t st = as_stream(stream);
  auto into = [&](uint32_t* wt, uint16_t* stl, int row0, int N, int K, int Ntot) -> w4a8_status {
    W4A8_CUDA_TRY(repack_run(w_p2, s_p2, N, K, Ntot, row0, wt, stl, st));
    return W4A8_OK;
  };
  const int QKV = m->qkv_rows;
  if (kind >= W4A8_T_Q && kind <= W4A8_T_DOWN && (layer < 0 || layer >= d.n_layers)) return W4A8_ERR_ARG;
  switch (kind) {
    case W4A8_T_Q: return into(m->qkv_w[layer], m->qkv_s[layer], 0, QD, H, QKV);
    case W4A8_T_K: return into(m->qkv_w[layer], m->qkv_s[layer], QD, KVD, H, QKV);
    case W4A8_T_V: return into(m->qkv_w[layer], m->qkv_s[layer], QD + KVD, KVD, H, QKV);
    case W4A8_T_O: return into(m->o_w[layer], m->o_s[layer], 0, H, QD, H);
    case W4A8_T_GATE: return into(m->gu_w[layer], m->gu_s[layer], 0, F, H, 2 * F);
    case W4A8_T_UP: return into(m->gu_w[layer], m->gu_s[layer], F, F, H, 2 * F);
    case W4A8_T_DOWN: return into(m->dn_w[layer], m->dn_s[layer], 0, H, F, H);
    case W4A8_T_EMBED: {
      W4A8_CUDA_TRY(cudaMemcpyAsync(m->emb_w, w_p2, (size_t)d.V * H / 2, cudaMemcpyDeviceToDevice, st));
      W4A8_CUDA_TRY(cudaMemcpyAsync(m->emb_s, s_p2, (size_t)d.V * H / 16, cudaMemcpyDeviceToDevice, st));
      if (d.tied) return into(m->lm_w, m->lm_s, 0, d.V, H, d.V);
      return W4A8_OK;
    }
    case W4A8_T_LM_HEAD:
      if (d.tied) return W4A8_ERR_ARG;
      return into(m->lm_w, m->lm_s, 0, d.V, H, d.V);
    default: return W4A8_ERR_ARG;
  }
}

W4A8_API w4a8_status w4a8_model_weight_bytes(const w4a8_model* m, size_t* bytes) {
  if (!m || !bytes) return W4A8_ERR_ARG;
  *bytes = m->bytes;
  return W4A8_OK;
}

W4A8_API void w4a8_model_destroy(w4a8_model* m) { delete m; }

// ---------------------------------------------------------------------------- session

W4A8_API w4a8_status w4a8_session_create(w4a8_model* m, const w4a8_session_desc* desc, w4a8_session** out) {
  if (!m || !desc || !out) return W4A8_ERR_ARG;
  if (desc->kv_cap < kMaxWidth + 1 || desc->ctx_cap < kMaxCont + 2 || desc->max_window < 1 ||
      desc->max_window > kMaxWindow)
    return W4A8_ERR_ARG;
  if (desc->mem_cap < 0 || desc->mem_cap > kMaxMemory) return W4A8_ERR_ARG;
  // the drafter keeps one byte per scanned position (context and memory) in shared memory
  if (desc->ctx_cap > 200 * 1024 || desc->ctx_cap + desc->mem_cap > 220 * 1024) return W4A8_ERR_CAPACITY;
  const ModelDims& d = m->d;
  w4a8_session* s = new (std::nothrow) w4a8_session();
  if (!s) return W4A8_ERR_NOMEM;
  s->m = m;
  s->max_window = desc->max_window;
  DecoderBufs& b = s->b;
  b.kv_cap = desc->kv_cap;
  b.ctx_cap = desc->ctx_cap;
  b.n_chunks = (desc->kv_cap + kAttnChunk - 1) / kAttnChunk;
  b.max_window = desc->max_window;
  b.eos_id = desc->eos_id;
  b.mem_cap = desc->mem_cap;
  const int Kmax = std::max(std::max(d.H, d.F), d.Hq * d.D);
  // per-slice outputs of the projections (EPI_PARTIAL)
  size_t part = std::max({mm_partial_floats(m->p_lm), mm_partial_floats(m->p_qkv), mm_partial_floats(m->p_o),
                          mm_partial_floats(m->p_gu), mm_partial_floats(m->p_dn)});
  int tick = std::max({m->p_qkv.n_rg, m->p_o.n_rg, m->p_gu.n_rg, m->p_dn.n_rg, m->p_lm.n_rg});
  const size_t kv = (size_t)d.n_layers * d.Hkv * desc->kv_cap * d.D * sizeof(float);
  Arena& A = s->arena;
  constexpr int kChains = kMaxBucket / kMaxWidth;  // attention chains of a prefill bucket
  const int QD = d.Hq * d.D;
  bool ok = A.dalloc(&b.ctl, sizeof(SpecCtl)) && A.dalloc(&b.tree, sizeof(TreeState)) &&
            A.dalloc(&b.rec, sizeof(AcceptRec)) && A.dalloc(&b.ctx, (size_t)desc->ctx_cap * 4) &&
            A.dalloc(&b.pred, kMaxWidth * 4) && A.dalloc(&b.x, (size_t)kMaxBucket * d.H * 4) &&
            A.dalloc(&b.qkv, (size_t)kMaxBucket * std::max(m->qkv_rows, QD) * 4) &&
            A.dalloc(&b.qrot, (size_t)kMaxBucket * QD * 4) && A.dalloc(&b.gu, (size_t)kMaxBucket * 2 * d.F * 4) &&
            A.dalloc(&b.o_part, (size_t)kChains * b.n_chunks * kMaxWidth * QD * 4) &&
            A.dalloc(&b.ml_part, (size_t)kChains * b.n_chunks * kMaxWidth * d.Hq * 8) &&
            A.dalloc(&b.act, act_bytes_nt(Kmax, act_tiles(kMaxBucket))) &&
            A.dalloc(&b.a_s, kMaxBucket * 4) && A.dalloc(&b.mm_part, part * 4) && A.dalloc(&b.tickets, (size_t)tick * 4) &&
            A.dalloc(&b.kcache, kv) && A.dalloc(&b.vcache, kv) &&
            A.dalloc(&b.rope, (size_t)desc->kv_cap * (d.D / 2) * sizeof(float2)) &&
            A.dalloc(&b.qpart, (size_t)kMaxBucket * (std::max({d.H, d.F, QD}) / 512 + d.Hq + 2) * sizeof(float2)) &&
            A.dalloc(&b.argmax_part, (size_t)kMaxWidth * ((d.V + 8191) / 8192) * sizeof(float2)) &&
            A.dalloc(&b.argmax_tickets, kMaxWidth * 4) && A.dalloc(&b.attn_tickets, (size_t)kChains * d.Hkv * 4) &&
            A.dalloc(&b.mem, (size_t)std::max(desc->mem_cap, 1) * 4) && A.dalloc(&b.mem_len, sizeof(int)) &&
            A.dalloc(&b.wstats, (size_t)desc->max_window * sizeof(StepStats)) &&
            A.dalloc(&b.wtok, (size_t)desc->max_window * kMaxWidth * 4) &&
            A.dalloc(&s->dev_rec, kRecBytesFixed + (size_t)desc->max_window * kRecStepBytes) &&
            A.dalloc(&s->prompt_dev, (size_t)desc->ctx_cap * 4) &&
            A.halloc(&s->host_rec[0], kRecBytesFixed + (size_t)desc->max_window * kRecStepBytes) &&
            A.halloc(&s->host_rec[1], kRecBytesFixed + (size_t)desc->max_window * kRecStepBytes) &&
            A.halloc(&s->pin, (size_t)std::max(desc->ctx_cap, 4096) * 4);
  if (!ok) {
    delete s;
    return W4A8_ERR_NOMEM;
  }
  // zero everything that is read before written (fragment padding groups, tickets, records)
  cudaError_t e = cudaSuccess;
  e = e == cudaSuccess ? cudaMemset(b.act, 0, act_bytes_nt(Kmax, act_tiles(kMaxBucket))) : e;
  e = e == cudaSuccess ? cudaMemset(b.tickets, 0, (size_t)tick * 4) : e;
  e = e == cudaSuccess ? cudaMemset(b.argmax_tickets, 0, kMaxWidth * 4) : e;
  e = e == cudaSuccess ? cudaMemset(b.attn_tickets, 0, (size_t)kChains * d.Hkv * 4) : e;
  e = e == cudaSuccess ? cudaMemset(b.ctl, 0, sizeof(SpecCtl)) : e;
  e = e == cudaSuccess ? cudaMemset(b.rec, 0, sizeof(AcceptRec)) : e;
  e = e == cudaSuccess ? cudaMemset(b.mem_len, 0, sizeof(int)) : e;
  e = e == cudaSuccess ? cudaMemset(b.tree, 0, sizeof(TreeState)) : e;
  e = e == cudaSuccess ? cudaMemset(b.kcache, 0, kv) : e;
  e = e == cudaSuccess ? cudaMemset(b.vcache, 0, kv) : e;
  // RoPE table in double, rounded to fp32: (cos, sin)(pos * base^(-2j/D))
  std::vector<float2> rope((size_t)desc->kv_cap * (d.D / 2));
  for (int p = 0; p < desc->kv_cap; ++p)
    for (int j = 0; j < d.D / 2; ++j) {
      const double th = std::pow((double)d.rope_base, -2.0 * j / d.D);
      rope[(size_t)p * (d.D / 2) + j] = make_float2((float)std::cos(p * th), (float)std::sin(p * th));
    }
  e = e == cudaSuccess ? cudaMemcpy(b.rope, rope.data(), rope.size() * sizeof(float2), cudaMemcpyHostToDevice) : e;
  e = e == cudaSuccess ? cudaEventCreateWithFlags(&s->ev[0], cudaEventDisableTiming) : e;
  e = e == cudaSuccess ? cudaEventCreateWithFlags(&s->ev[1], cudaEventDisableTiming) : e;
  e = e == cudaSuccess ? cudaStreamCreateWithFlags(&s->cap, cudaStreamNonBlocking) : e;
  e = e == cudaSuccess ? attn_configure(d, attn_smem_bytes(d.D, kMaxWidth * (d.Hq / d.Hkv))) : e;
  e = e == cudaSuccess ? attn_tensor_maps(b, d) : e;
  e = e == cudaSuccess ? mm_configure() : e;
  e = e == cudaSuccess ? draft_configure(desc->ctx_cap + desc->mem_cap) : e;
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    delete s;
    return W4A8_ERR_CUDA;
  }
  *out = s;
  return W4A8_OK;
}

W4A8_API void w4a8_session_destroy(w4a8_session* s) {
  if (s) cudaDeviceSynchronize();
  delete s;
}

namespace {
bool d_ok_for_buckets(const ModelDims& d) { return d.Hq / d.Hkv >= 2; }
}  // namespace

W4A8_API w4a8_status w4a8_prefill(w4a8_session* s, const int32_t* prompt, int n, int max_new, void* stream) {
  if (!s || !prompt || n < 1 || max_new < 0) return W4A8_ERR_ARG;
  if (!s->q.empty()) return W4A8_ERR_ARG;
  const DecoderBufs& b = s->b;
  if ((long long)n + max_new + kMaxCont + 1 > b.ctx_cap) return W4A8_ERR_CAPACITY;
  if ((long long)n + max_new + kMaxWidth > b.kv_cap) return W4A8_ERR_CAPACITY;
  cudaStream_t st = as_stream(stream);
  W4A8_CUDA_TRY(cudaMemcpyAsync(b.ctx, prompt, (size_t)n * 4, cudaMemcpyDeviceToDevice, st));
  W4A8_CUDA_TRY(launch_pdl(k_init_ctl, dim3(1), dim3(32), 0, st, b.ctl, b.rec, (const int32_t*)b.ctx, n, max_new));
  // Integer prefill in wide buckets [P1 Small-Batch Verification Kernels (token buckets);
  // Experiments: request latency]: full buckets of kMaxBucket (64) prompt tokens replay one
  // captured graph (the kernels read their position from the control word): the matmuls and the
  // row-wise kernels take the whole bucket, the attention its four chains of kMaxWidth.  Two or
  // three whole chains left over run as one such pass, the rest as one chain of fewer nodes.
  // Every step of a token's forward is row-local with the same order, so the cache holds the
  // bits of sequential steps.
  // (models whose query heads do not share KV heads keep chains of kMaxWidth: their attention
  // merges inside the chunk kernel, which takes one chain per launch)
  const int buckets = d_ok_for_buckets(s->m->d) ? (n - 1) / kMaxBucket : 0;
  if (buckets > 0 && !s->bucket_graph) {
    cudaGraph_t g = nullptr;
    W4A8_CUDA_TRY(cudaStreamBeginCapture(s->cap, cudaStreamCaptureModeThreadLocal));
    cudaError_t e = launch_chain_tree(b, 0, kMaxWidth, s->cap);
    if (e == cudaSuccess) e = forward(s, kMaxBucket, false, nullptr, s->cap, nullptr, true);
    if (e == cudaSuccess) e = launch_commit_chain(b, kMaxBucket, s->cap);
    const cudaError_t e2 = cudaStreamEndCapture(s->cap, &g);
    if (e == cudaSuccess) e = e2;
    if (e == cudaSuccess) e = cudaGraphInstantiate(&s->bucket_graph, g, 0);
    if (g) cudaGraphDestroy(g);
    if (e != cudaSuccess) {
      s->bucket_graph = nullptr;
      (void)cudaGetLastError();
      return W4A8_ERR_CUDA;
    }
  }
  for (int c = 0; c < buckets; ++c) W4A8_CUDA_TRY(cudaGraphLaunch(s->bucket_graph, st));
  int done = buckets * kMaxBucket;
  // two or three whole chains left: one pass over them, as in a bucket (not captured)
  const int whole = d_ok_for_buckets(s->m->d) ? ((n - 1 - done) / kMaxWidth) * kMaxWidth : 0;
  if (whole >= 2 * kMaxWidth) {
    W4A8_CUDA_TRY(launch_chain_tree(b, 0, kMaxWidth, st));
    W4A8_CUDA_TRY(forward(s, whole, false, nullptr, st, nullptr, true));
    W4A8_CUDA_TRY(launch_commit_chain(b, whole, st));
    done += whole;
  }
  while (done < n - 1) {
    const int len = std::min(kMaxWidth, n - 1 - done);
    W4A8_CUDA_TRY(launch_chain_tree(b, done, len, st));
    W4A8_CUDA_TRY(forward(s, len, false, nullptr, st));
    W4A8_CUDA_TRY(launch_commit_chain(b, len, st));
    done += len;
  }
  W4A8_CUDA_TRY(launch_draft(b, 1, st));
  return W4A8_OK;
}

W4A8_API w4a8_status tree_verify_step(w4a8_session* s, int N, float* logits, void* stream) {
  if (!s || N < 1 || N > kMaxWidth) return W4A8_ERR_ARG;
  W4A8_CUDA_TRY(forward(s, N, true, logits, as_stream(stream)));
  return W4A8_OK;
}

W4A8_API w4a8_status w4a8_model_trace_bytes(const w4a8_model* m, int N, size_t* bytes) {
  if (!m || !bytes || N < 1 || N > kMaxWidth) return W4A8_ERR_ARG;
  *bytes = trace_bytes(m->d, N);
  return W4A8_OK;
}

W4A8_API w4a8_status w4a8_tree_verify_trace(w4a8_session* s, int N, float* logits, int8_t* codes, size_t codes_bytes,
                                            void* stream) {
  if (!s || !codes || N < 1 || N > kMaxWidth) return W4A8_ERR_ARG;
  if (codes_bytes < trace_bytes(s->m->d, N)) return W4A8_ERR_CAPACITY;
  W4A8_CUDA_TRY(forward(s, N, true, logits, as_stream(stream), codes));
  return W4A8_OK;
}

W4A8_API w4a8_status accept_greedy(w4a8_session* s, int N, void* stream) {
  if (!s || N < 1 || N > kMaxWidth) return W4A8_ERR_ARG;
  W4A8_CUDA_TRY(launch_accept(s->b, N, 0, as_stream(stream)));
  return W4A8_OK;
}

W4A8_API w4a8_status kv_compact(w4a8_session* s, void* stream) {
  if (!s) return W4A8_ERR_ARG;
  W4A8_CUDA_TRY(launch_compact(s->b, s->m->d, as_stream(stream)));
  return W4A8_OK;
}

W4A8_API w4a8_status ngram_draft(w4a8_session* s, void* stream) {
  if (!s) return W4A8_ERR_ARG;
  W4A8_CUDA_TRY(launch_draft(s->b, 1, as_stream(stream)));
  return W4A8_OK;
}

W4A8_API w4a8_status w4a8_spec_step(w4a8_session* s, int N, void* stream) {
  if (!s || N < 1 || N > kMaxWidth) return W4A8_ERR_ARG;
  W4A8_CUDA_TRY(step(s, N, 0, as_stream(stream)));
  return W4A8_OK;
}

namespace {
w4a8_status window_graph(w4a8_session* s, int N, int W, int slot, cudaGraphExec_t* out) {
  const long long key = graph_key(N, W, slot);
  auto it = s->graphs.find(key);
  if (it != s->graphs.end()) {
    *out = it->second;
    return W4A8_OK;
  }
  cudaGraph_t g = nullptr;
  W4A8_CUDA_TRY(cudaStreamBeginCapture(s->cap, cudaStreamCaptureModeThreadLocal));
  cudaError_t e = cudaSuccess;
  for (int k = 0; k < W && e == cudaSuccess; ++k) e = step(s, N, k, s->cap);
  if (e == cudaSuccess)
    e = launch_pdl(k_window_close, dim3(1), dim3(256), 0, s->cap, (const SpecCtl*)s->b.ctl,
                   (const StepStats*)s->b.wstats, (const int32_t*)s->b.wtok, W, s->dev_rec);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(s->host_rec[slot], s->dev_rec, kRecBytesFixed + (size_t)W * kRecStepBytes,
                        cudaMemcpyDeviceToHost, s->cap);
  cudaError_t e2 = cudaStreamEndCapture(s->cap, &g);
  if (e != cudaSuccess || e2 != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    (void)cudaGetLastError();
    return W4A8_ERR_CUDA;
  }
  size_t n_nodes = 0;
  int n_kernels = 0;
  if (cudaGraphGetNodes(g, nullptr, &n_nodes) == cudaSuccess && n_nodes > 0) {
    std::vector<cudaGraphNode_t> nodes(n_nodes);
    if (cudaGraphGetNodes(g, nodes.data(), &n_nodes) == cudaSuccess)
      for (size_t i = 0; i < n_nodes; ++i) {
        cudaGraphNodeType t;
        if (cudaGraphNodeGetType(nodes[i], &t) == cudaSuccess && t == cudaGraphNodeTypeKernel) ++n_kernels;
      }
  }
  cudaGraphExec_t ge = nullptr;
  e = cudaGraphInstantiate(&ge, g, 0);
  cudaGraphDestroy(g);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return W4A8_ERR_CUDA;
  }
  s->graphs[key] = ge;
  s->graph_kernels[key] = n_kernels;
  *out = ge;
  return W4A8_OK;
}
}  // namespace

W4A8_API w4a8_status spec_window(w4a8_session* s, int N, int W, void* stream) {
  if (!s || N < 1 || N > kMaxWidth || W < 1 || W > s->max_window) return W4A8_ERR_ARG;
  if (s->q.size() >= 2) return W4A8_ERR_ARG;
  const int slot = s->next_slot;
  cudaGraphExec_t ge = nullptr;
  w4a8_status st = window_graph(s, N, W, slot, &ge);
  if (st != W4A8_OK) return st;
  cudaStream_t cs = as_stream(stream);
  W4A8_CUDA_TRY(cudaGraphLaunch(ge, cs));
  W4A8_CUDA_TRY(cudaEventRecord(s->ev[slot], cs));
  s->kernels += s->graph_kernels[graph_key(N, W, slot)];
  s->q.push_back({slot, W, N});
  s->next_slot ^= 1;
  return W4A8_OK;
}

W4A8_API w4a8_status spec_poll(w4a8_session* s, w4a8_ctl16* ctl, w4a8_step_stats* stats, int* n_stats,
                               int32_t* tokens, int* n_tokens, int64_t timeout_us) {
  if (!s) return W4A8_ERR_ARG;
  if (s->q.empty()) return W4A8_ERR_ARG;
  const w4a8_session::Flight f = s->q.front();
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    const cudaError_t e = cudaEventQuery(s->ev[f.slot]);
    if (e == cudaSuccess) break;
    if (e != cudaErrorNotReady) {
      (void)cudaGetLastError();
      return W4A8_ERR_CUDA;
    }
    if (timeout_us >= 0) {
      const auto us = std::chrono::duration_cast<std::chrono::microseconds>(std::chrono::steady_clock::now() - t0);
      if (us.count() > timeout_us) return W4A8_ERR_TIMEOUT;
    }
  }
  s->q.pop_front();
  s->host_syncs++;
  const uint8_t* r = s->host_rec[f.slot];
  SpecCtl c;
  std::memcpy(&c, r, sizeof(c));
  if (ctl) {
    ctl->committed_len = c.committed_len;
    ctl->n_generated = c.n_generated;
    ctl->flags = c.flags;
    ctl->root_tok = c.root_tok;
  }
  const StepStats* ss = reinterpret_cast<const StepStats*>(r + kRecBytesFixed);
  const int32_t* tk = reinterpret_cast<const int32_t*>(r + kRecBytesFixed + (size_t)f.W * sizeof(StepStats));
  int nt = 0;
  for (int k = 0; k < f.W; ++k) {
    if (stats) std::memcpy(&stats[k], &ss[k], sizeof(StepStats));
    for (int j = 0; j < ss[k].n_emitted; ++j) {
      if (tokens) tokens[nt] = tk[k * kMaxWidth + j];
      ++nt;
    }
  }
  if (n_stats) *n_stats = f.W;
  if (n_tokens) *n_tokens = nt;
  return W4A8_OK;
}

W4A8_API w4a8_status w4a8_calibrate(w4a8_session* s, const int* widths, int n_widths, int reps, int trials,
                                    float* t_us) {
  if (!s || !widths || !t_us || n_widths <= 0 || reps <= 0 || trials <= 0) return W4A8_ERR_ARG;
  if (!s->q.empty()) return W4A8_ERR_ARG;
  SpecCtl c;
  w4a8_status st = sync_read(s, &c, s->b.ctl, sizeof(c));
  if (st != W4A8_OK) return st;
  if (c.flags & FLAG_STOP_MASK) return W4A8_ERR_DEVICE_FLAG;
  cudaStream_t cs = s->cap;
  cudaEvent_t e0, e1;
  W4A8_CUDA_TRY(cudaEventCreate(&e0));
  W4A8_CUDA_TRY(cudaEventCreate(&e1));
  w4a8_status res = W4A8_OK;
  for (int i = 0; i < n_widths && res == W4A8_OK; ++i) {
    const int N = widths[i];
    if (N < 1 || N > kMaxWidth || c.committed_len + N > (uint32_t)s->b.kv_cap) {
      res = W4A8_ERR_ARG;
      break;
    }
    cudaGraph_t g = nullptr;
    cudaGraphExec_t ge = nullptr;
    cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
      // verification pass + drafting: leaves the committed state unchanged
      cudaError_t e3 = forward(s, N, true, nullptr, cs);
      if (e3 == cudaSuccess) e3 = launch_draft(s->b, 1, cs);
      e = cudaStreamEndCapture(cs, &g);
      if (e == cudaSuccess) e = e3;
    }
    if (e == cudaSuccess) e = cudaGraphInstantiate(&ge, g, 0);
    std::vector<float> ts;
    if (e == cudaSuccess) e = cudaGraphLaunch(ge, cs);
    for (int t = 0; t < trials && e == cudaSuccess; ++t) {
      e = cudaEventRecord(e0, cs);
      for (int r = 0; r < reps && e == cudaSuccess; ++r) e = cudaGraphLaunch(ge, cs);
      if (e == cudaSuccess) e = cudaEventRecord(e1, cs);
      if (e == cudaSuccess) e = cudaEventSynchronize(e1);
      float ms = 0.0f;
      if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
      ts.push_back(ms * 1000.0f / reps);
    }
    if (ge) cudaGraphExecDestroy(ge);
    if (g) cudaGraphDestroy(g);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      res = W4A8_ERR_CUDA;
      break;
    }
    std::sort(ts.begin(), ts.end());
    const size_t n = ts.size();
    t_us[i] = (n % 2) ? ts[n / 2] : 0.5f * (ts[n / 2 - 1] + ts[n / 2]);
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return res;
}

W4A8_API w4a8_status w4a8_generate(w4a8_session* s, const w4a8_decode_opts* o, int32_t* out, int* n_out,
                                   w4a8_decode_report* rep, void* stream) {
  if (!s || !o || !out || !n_out) return W4A8_ERR_ARG;
  if (o->window < 1 || o->window > s->max_window || o->in_flight < 1 || o->in_flight > 2) return W4A8_ERR_ARG;
  if (o->fixed_width < 0 || o->fixed_width > kMaxWidth) return W4A8_ERR_ARG;
  if (!s->q.empty()) return W4A8_ERR_ARG;
  SpecCtl c0;
  w4a8_status st = W4A8_OK;
  W4A8_CUDA_TRY(cudaStreamSynchronize(as_stream(stream)));
  st = sync_read(s, &c0, s->b.ctl, sizeof(c0));
  if (st != W4A8_OK) return st;
  const int max_new = (int)(c0.max_new - c0.n_generated);
  w4a8_controller* ctrl = nullptr;
  if (o->fixed_width == 0) {
    st = w4a8_controller_create(o->widths, o->t_us, o->n_widths, &ctrl);
    if (st != W4A8_OK) return st;
  }
  w4a8_decode_report r;
  std::memset(&r, 0, sizeof(r));
  const long long syncs0 = s->host_syncs, kernels0 = s->kernels;
  std::vector<w4a8_step_stats> stats((size_t)o->window);
  std::vector<int32_t> toks((size_t)o->window * kMaxWidth);
  int produced = 0;
  bool done = (c0.flags & FLAG_STOP_MASK) != 0 || max_new <= 0, have_t = false;
  uint32_t t_prev = 0, t_first = 0, t_last = 0;
  w4a8_ctl16 c16 = {c0.committed_len, c0.n_generated, c0.flags, c0.root_tok};
  auto launch_one = [&]() -> w4a8_status {
    const int N = ctrl ? w4a8_controller_choose(ctrl) : o->fixed_width;
    return spec_window(s, N, o->window, stream);
  };
  for (int i = 0; i < o->in_flight && !done && st == W4A8_OK; ++i) st = launch_one();
  while (st == W4A8_OK && !s->q.empty()) {
    const int N = s->q.front().N;
    int ns = 0, nt = 0;
    st = spec_poll(s, &c16, stats.data(), &ns, toks.data(), &nt, o->timeout_us);
    if (st != W4A8_OK) break;
    r.n_windows++;
    for (int j = 0; j < nt && produced < max_new; ++j) out[produced++] = toks[j];
    int executed = 0;
    for (int k = 0; k < ns; ++k) {
      if (stats[k].n_emitted == 0) continue;
      ++executed;
      r.n_steps++;
      r.width_steps[N]++;
      r.accepted_drafts += stats[k].n_accepted_drafts;
      if (!have_t) {
        t_first = stats[k].t_lo;
        have_t = true;
      }
      t_last = stats[k].t_lo;
    }
    if (ctrl && executed > 0) {
      double interval = 0.0;
      if (r.n_windows > 1) interval = (double)(uint32_t)(stats[executed - 1].t_lo - t_prev) * 1e-3;
      w4a8_controller_observe(ctrl, N, stats.data(), executed, interval);
    }
    if (executed > 0) t_prev = stats[executed - 1].t_lo;
    if (c16.flags & FLAG_STOP_MASK) done = true;
    if (!done) st = launch_one();
  }
  while (!s->q.empty()) {  // leave no window in flight
    w4a8_status s2 = spec_poll(s, nullptr, nullptr, nullptr, nullptr, nullptr, o->timeout_us);
    if (s2 != W4A8_OK) {
      if (st == W4A8_OK) st = s2;
      break;
    }
  }
  if (ctrl) w4a8_controller_destroy(ctrl);
  r.n_tokens = produced;
  r.flags = c16.flags;
  r.host_syncs = (int)(s->host_syncs - syncs0);
  r.kernels = s->kernels - kernels0;
  r.device_us = have_t ? (double)(uint32_t)(t_last - t_first) * 1e-3 : 0.0;
  *n_out = produced;
  if (rep) *rep = r;
  if (st != W4A8_OK) return st;
  return (c16.flags & FLAG_ERR_MASK) ? W4A8_ERR_DEVICE_FLAG : W4A8_OK;
}

W4A8_API w4a8_status w4a8_decode(w4a8_session* s, const int32_t* prompt, int n_prompt, const w4a8_decode_opts* o,
                                 int32_t* out, int* n_out, w4a8_decode_report* rep, void* stream) {
  if (!s || !prompt || !o || !out || !n_out || n_prompt < 1) return W4A8_ERR_ARG;
  if (n_prompt > s->b.ctx_cap) return W4A8_ERR_CAPACITY;
  if (!s->q.empty()) return W4A8_ERR_ARG;
  cudaStream_t cs = as_stream(stream);
  W4A8_CUDA_TRY(cudaStreamSynchronize(cs));
  std::memcpy(s->pin, prompt, (size_t)n_prompt * 4);
  W4A8_CUDA_TRY(cudaMemcpyAsync(s->prompt_dev, s->pin, (size_t)n_prompt * 4, cudaMemcpyHostToDevice, cs));
  w4a8_status st = w4a8_prefill(s, s->prompt_dev, n_prompt, o->max_new, stream);
  if (st != W4A8_OK) return st;
  return w4a8_generate(s, o, out, n_out, rep, stream);
}

W4A8_API w4a8_status w4a8_time_matmuls(w4a8_session* s, int N, int reps, double* us_per_launch,
                                       double* bytes_per_launch, int* launches_per_pass) {
  if (!s || N < 1 || N > kMaxWidth || reps < 1 || !us_per_launch || !bytes_per_launch) return W4A8_ERR_ARG;
  if (!s->q.empty()) return W4A8_ERR_ARG;
  w4a8_model* m = s->m;
  const ModelDims& d = m->d;
  const DecoderBufs& b = s->b;
  unsigned* flags = &b.ctl->flags;
  SpecCtl c;
  w4a8_status st = sync_read(s, &c, b.ctl, sizeof(c));
  if (st != W4A8_OK) return st;
  if (c.flags & FLAG_STOP_MASK) return W4A8_ERR_DEVICE_FLAG;  // stopped kernels would do no work
  auto mbytes = [&](const MatmulPlan& p) {
    return 0.5 * p.N * p.K + 2.0 * p.N * (p.K / 32) + (double)N * p.K + 4.0 * N + 4.0 * N * p.N;
  };
  double bytes = 0.0;
  int launches = 0;
  cudaStream_t cs = s->cap;
  cudaGraph_t g = nullptr;
  cudaGraphExec_t ge = nullptr;
  cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  cudaError_t e3 = cudaSuccess;
  for (int l = 0; l < d.n_layers && e3 == cudaSuccess && e == cudaSuccess; ++l) {
    e3 = mm_run(m->p_qkv, m->qkv_w[l], m->qkv_s[l], b.act, b.a_s, N, nullptr, 0, EPI_PARTIAL, b.mm_part, b.tickets,
                flags, flags, cs);
    if (e3 == cudaSuccess)
      e3 = mm_run(m->p_o, m->o_w[l], m->o_s[l], b.act, b.a_s, N, nullptr, 0, EPI_PARTIAL, b.mm_part, b.tickets,
                  flags, flags, cs);
    if (e3 == cudaSuccess)
      e3 = mm_run(m->p_gu, m->gu_w[l], m->gu_s[l], b.act, b.a_s, N, nullptr, 0, EPI_PARTIAL, b.mm_part, b.tickets,
                  flags, flags, cs);
    if (e3 == cudaSuccess)
      e3 = mm_run(m->p_dn, m->dn_w[l], m->dn_s[l], b.act, b.a_s, N, nullptr, 0, EPI_PARTIAL, b.mm_part, b.tickets,
                  flags, flags, cs);
    bytes += mbytes(m->p_qkv) + mbytes(m->p_o) + mbytes(m->p_gu) + mbytes(m->p_dn);
    launches += 4;
  }
  if (e3 == cudaSuccess)
    e3 = mm_run(m->p_lm, m->lm_w, m->lm_s, b.act, b.a_s, N, nullptr, 0, EPI_PARTIAL, b.mm_part, b.tickets, flags,
                flags, cs);
  bytes += mbytes(m->p_lm);
  launches += 1;
  if (e == cudaSuccess) e = cudaStreamEndCapture(cs, &g);
  if (e == cudaSuccess) e = e3;
  if (e == cudaSuccess) e = cudaGraphInstantiate(&ge, g, 0);
  cudaEvent_t a = nullptr, z = nullptr;
  if (e == cudaSuccess) e = cudaEventCreate(&a);
  if (e == cudaSuccess) e = cudaEventCreate(&z);
  if (e == cudaSuccess) e = cudaGraphLaunch(ge, cs);
  if (e == cudaSuccess) e = cudaEventRecord(a, cs);
  for (int r = 0; r < reps && e == cudaSuccess; ++r) e = cudaGraphLaunch(ge, cs);
  if (e == cudaSuccess) e = cudaEventRecord(z, cs);
  if (e == cudaSuccess) e = cudaEventSynchronize(z);
  float ms = 0.0f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, a, z);
  if (a) cudaEventDestroy(a);
  if (z) cudaEventDestroy(z);
  if (ge) cudaGraphExecDestroy(ge);
  if (g) cudaGraphDestroy(g);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return W4A8_ERR_CUDA;
  }
  *us_per_launch = (double)ms * 1000.0 / ((double)reps * launches);
  *bytes_per_launch = bytes / launches;
  if (launches_per_pass) *launches_per_pass = launches;
  return W4A8_OK;
}

namespace {
__global__ void k_raise_flags(SpecCtl* ctl, uint32_t f) {
  griddep_enter();
  if (threadIdx.x == 0) atomicOr(&ctl->flags, f);
}
}  // namespace

W4A8_API w4a8_status w4a8_session_raise_flags(w4a8_session* s, uint32_t flags, void* stream) {
  if (!s || (flags & ~(uint32_t)FLAG_STOP_MASK)) return W4A8_ERR_ARG;
  W4A8_CUDA_TRY(launch_pdl(k_raise_flags, dim3(1), dim3(32), 0, as_stream(stream), s->b.ctl, flags));
  return W4A8_OK;
}

// ------------------------------------------------------------------ state access (sync)

W4A8_API w4a8_status w4a8_session_get_ctl(w4a8_session* s, w4a8_ctl* ctl) {
  if (!s || !ctl) return W4A8_ERR_ARG;
  W4A8_CUDA_TRY(cudaDeviceSynchronize());
  return sync_read(s, ctl, s->b.ctl, sizeof(SpecCtl));
}

W4A8_API w4a8_status w4a8_session_set_tree(w4a8_session* s, const int32_t* tok, const int32_t* parent, int n) {
  if (!s || !tok || !parent || n < 1 || n > kMaxWidth) return W4A8_ERR_ARG;
  if (parent[0] != -1) return W4A8_ERR_ARG;
  TreeState t;
  std::memset(&t, 0, sizeof(t));
  for (int i = 0; i < kMaxWidth; ++i) {
    if (i < n) {
      if (i > 0 && (parent[i] < 0 || parent[i] >= i)) return W4A8_ERR_ARG;
      if (tok[i] < 0 || tok[i] >= s->m->d.V) return W4A8_ERR_ARG;
      t.tok[i] = tok[i];
      t.parent[i] = parent[i];
      t.depth[i] = i == 0 ? 0 : t.depth[parent[i]] + 1;
    } else {
      t.tok[i] = 0;
      t.parent[i] = 0;
      t.depth[i] = 1;
    }
  }
  t.n_valid = n;
  t.best_len = 0;
  W4A8_CUDA_TRY(cudaDeviceSynchronize());
  W4A8_CUDA_TRY(cudaMemcpy(s->b.tree, &t, sizeof(t), cudaMemcpyHostToDevice));
  const uint32_t nv = (uint32_t)n;
  W4A8_CUDA_TRY(cudaMemcpy(&s->b.ctl->n_valid, &nv, 4, cudaMemcpyHostToDevice));
  return W4A8_OK;
}

W4A8_API w4a8_status w4a8_session_get_tree(w4a8_session* s, int32_t* tok, int32_t* parent, int32_t* depth,
                                           int* n_valid, int* best_len) {
  if (!s) return W4A8_ERR_ARG;
  W4A8_CUDA_TRY(cudaDeviceSynchronize());
  TreeState t;
  w4a8_status st = sync_read(s, &t, s->b.tree, sizeof(t));
  if (st != W4A8_OK) return st;
  for (int i = 0; i < kMaxWidth; ++i) {
    if (tok) tok[i] = t.tok[i];
    if (parent) parent[i] = t.parent[i];
    if (depth) depth[i] = t.depth[i];
  }
  if (n_valid) *n_valid = t.n_valid;
  if (best_len) *best_len = t.best_len;
  return W4A8_OK;
}

W4A8_API w4a8_status w4a8_session_get_pred(w4a8_session* s, int32_t* pred, int n) {
  if (!s || !pred || n < 1 || n > kMaxWidth) return W4A8_ERR_ARG;
  W4A8_CUDA_TRY(cudaDeviceSynchronize());
  return sync_read(s, pred, s->b.pred, (size_t)n * 4);
}

W4A8_API w4a8_status w4a8_session_get_context(w4a8_session* s, int32_t* out, int cap, int* n) {
  if (!s || !out || !n || cap < 0) return W4A8_ERR_ARG;
  W4A8_CUDA_TRY(cudaDeviceSynchronize());
  SpecCtl c;
  w4a8_status st = sync_read(s, &c, s->b.ctl, sizeof(c));
  if (st != W4A8_OK) return st;
  *n = (int)c.ctx_len;
  const int k = std::min(cap, (int)c.ctx_len);
  if (k > 0) return sync_read(s, out, s->b.ctx, (size_t)k * 4);
  return W4A8_OK;
}

W4A8_API w4a8_status w4a8_session_memory_append(w4a8_session* s, const int32_t* tokens, int n) {
  if (!s || (!tokens && n > 0) || n < 0) return W4A8_ERR_ARG;
  if (!s->q.empty()) return W4A8_ERR_ARG;
  const int cap = s->b.mem_cap;
  if (cap < 2) return W4A8_ERR_CAPACITY;
  for (int i = 0; i < n; ++i)
    if (tokens[i] < 0 || tokens[i] >= s->m->d.V) return W4A8_ERR_ARG;
  // an output longer than the memory keeps its last cap - 1 tokens; whole outputs are dropped
  // from the oldest until the new one fits
  const int keep = std::min(n, cap - 1);
  std::vector<int32_t>& mh = s->mem_host;
  while (!mh.empty() && (int)mh.size() + keep + 1 > cap) {
    size_t nxt = 1;
    while (nxt < mh.size() && mh[nxt] != -1) ++nxt;
    mh.erase(mh.begin(), mh.begin() + (long)nxt);
  }
  mh.push_back(-1);
  mh.insert(mh.end(), tokens + (n - keep), tokens + n);
  const int len = (int)mh.size();
  W4A8_CUDA_TRY(cudaDeviceSynchronize());
  W4A8_CUDA_TRY(cudaMemcpy(s->b.mem, mh.data(), (size_t)len * 4, cudaMemcpyHostToDevice));
  W4A8_CUDA_TRY(cudaMemcpy(s->b.mem_len, &len, sizeof(int), cudaMemcpyHostToDevice));
  return W4A8_OK;
}

W4A8_API w4a8_status w4a8_session_memory_clear(w4a8_session* s) {
  if (!s || !s->q.empty()) return W4A8_ERR_ARG;
  s->mem_host.clear();
  const int zero = 0;
  W4A8_CUDA_TRY(cudaDeviceSynchronize());
  W4A8_CUDA_TRY(cudaMemcpy(s->b.mem_len, &zero, sizeof(int), cudaMemcpyHostToDevice));
  return W4A8_OK;
}

W4A8_API w4a8_status w4a8_session_memory_get(const w4a8_session* s, int32_t* out, int cap, int* n) {
  if (!s || !n || cap < 0 || (!out && cap > 0)) return W4A8_ERR_ARG;
  *n = (int)s->mem_host.size();
  const int k = std::min(cap, *n);
  if (k > 0) std::memcpy(out, s->mem_host.data(), (size_t)k * 4);
  return W4A8_OK;
}

W4A8_API w4a8_status w4a8_session_attention(w4a8_session* s, int layer, int n, const float* q, float* out,
                                            void* stream) {
  if (!s || !q || !out || layer < 0 || layer >= s->m->d.n_layers || n < 1 || n > kMaxWidth) return W4A8_ERR_ARG;
  const ModelDims& d = s->m->d;
  cudaStream_t cs = as_stream(stream);
  // the kernel reads slots [0, committed_len + n): check the control state first
  W4A8_CUDA_TRY(cudaStreamSynchronize(cs));
  SpecCtl ctl;
  TreeState tree;
  W4A8_CUDA_TRY(cudaMemcpy(&ctl, s->b.ctl, sizeof(ctl), cudaMemcpyDeviceToHost));
  W4A8_CUDA_TRY(cudaMemcpy(&tree, s->b.tree, sizeof(tree), cudaMemcpyDeviceToHost));
  if ((ctl.flags & FLAG_STOP_MASK) != 0u) return W4A8_ERR_DEVICE_FLAG;
  if ((long long)ctl.committed_len + n > s->b.kv_cap) return W4A8_ERR_CAPACITY;
  if (n > tree.n_valid) return W4A8_ERR_ARG;
  const size_t qn = (size_t)n * d.Hq * d.D;
  W4A8_CUDA_TRY(cudaMemcpyAsync(s->b.qrot, q, qn * 4, cudaMemcpyDeviceToDevice, cs));
  W4A8_CUDA_TRY(launch_tree_attention(s->b, d, n, layer, cs));
  W4A8_CUDA_TRY(cudaMemcpyAsync(out, s->b.qkv, qn * 4, cudaMemcpyDeviceToDevice, cs));
  return W4A8_OK;
}

W4A8_API w4a8_status w4a8_session_load_kv(w4a8_session* s, int layer, int slot0, int n, const float* k_in,
                                          const float* v_in, void* stream) {
  if (!s || !k_in || !v_in || layer < 0 || layer >= s->m->d.n_layers || slot0 < 0 || n < 1 ||
      slot0 + n > s->b.kv_cap)
    return W4A8_ERR_ARG;
  const ModelDims& d = s->m->d;
  cudaStream_t cs = as_stream(stream);
  for (int h = 0; h < d.Hkv; ++h) {
    const size_t dst = (((size_t)layer * d.Hkv + h) * s->b.kv_cap + slot0) * d.D;
    const size_t src = (size_t)h * n * d.D;
    W4A8_CUDA_TRY(cudaMemcpyAsync(s->b.kcache + dst, k_in + src, (size_t)n * d.D * 4, cudaMemcpyDeviceToDevice, cs));
    W4A8_CUDA_TRY(cudaMemcpyAsync(s->b.vcache + dst, v_in + src, (size_t)n * d.D * 4, cudaMemcpyDeviceToDevice, cs));
  }
  return W4A8_OK;
}

W4A8_API w4a8_status w4a8_session_copy_kv(w4a8_session* s, int layer, int slot0, int n, float* k_out, float* v_out,
                                          void* stream) {
  if (!s || !k_out || !v_out || layer < 0 || layer >= s->m->d.n_layers || slot0 < 0 || n < 1 ||
      slot0 + n > s->b.kv_cap)
    return W4A8_ERR_ARG;
  const ModelDims& d = s->m->d;
  cudaStream_t cs = as_stream(stream);
  for (int h = 0; h < d.Hkv; ++h) {
    const size_t src = (((size_t)layer * d.Hkv + h) * s->b.kv_cap + slot0) * d.D;
    const size_t dst = (size_t)h * n * d.D;
    W4A8_CUDA_TRY(cudaMemcpyAsync(k_out + dst, s->b.kcache + src, (size_t)n * d.D * 4, cudaMemcpyDeviceToDevice, cs));
    W4A8_CUDA_TRY(cudaMemcpyAsync(v_out + dst, s->b.vcache + src, (size_t)n * d.D * 4, cudaMemcpyDeviceToDevice, cs));
  }
  return W4A8_OK;
}
