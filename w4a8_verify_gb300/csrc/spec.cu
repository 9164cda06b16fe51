// The GPU-resident speculation kernels: greedy acceptance, KV compaction, the suffix
// n-gram drafter and the chain trees of the prefill.
//
// "GPU-Resident Speculative Decoding ..." (Design > GPU-Resident Speculation Loop): an
// acceptance kernel walks the tree from the root and follows the child whose token equals
// the greedy prediction of its parent; the step commits the accepted drafts plus the token
// predicted after the last of them; a compaction kernel moves the keys and values of the
// accepted path into place; the drafter writes the next tree; generated tokens accumulate
// in a device buffer.  (Design > Draft-Free Drafting From Web Context): a parallel scan in
// which every context position computes the length of its match with the current suffix
// (orders up to 8), a selection of the best positions, and a single CTA that merges their
// continuations into a weighted trie and emits the most probable prefix-closed node set.
// "Exact Speculative And Assisted Decoding ..." (sections 4 and 7): greedy acceptance with
// a bonus token; commit and rollback move the logical KV length only.
#include "decoder.cuh"
#include "layers.cuh"

namespace w4a8 {

namespace {
__device__ __forceinline__ uint32_t globaltimer_lo() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return (uint32_t)t;
}
}  // namespace

// One warp.  pred[i] is the argmax of node i's logits.
__global__ void k_accept(SpecCtl* ctl, const TreeState* __restrict__ tree, const int32_t* __restrict__ pred, int N,
                         AcceptRec* rec, int32_t* ctx, int ctx_cap, int kv_cap, int max_width, StepStats* wstats,
                         int32_t* wtok, int wslot, int eos) {
  griddep_enter();
  const int lane = threadIdx.x;
  const uint32_t flags = ctl->flags;
  if (flags & FLAG_STOP_MASK) {
    if (lane == 0) {
      rec->valid = 0;
      StepStats z = {0, 0, 0, 0, globaltimer_lo()};
      wstats[wslot] = z;
    }
    return;
  }
  const int n_valid = min(tree->n_valid, N);
  const int my_tok = lane < kMaxWidth ? tree->tok[lane] : -1;
  const int my_par = lane < kMaxWidth ? tree->parent[lane] : -2;
  int path[kMaxWidth];
  path[0] = 0;
  int d = 0, cur = 0;
  while (d < kMaxWidth - 1) {
    const int target = pred[cur];
    const bool match = lane >= 1 && lane < n_valid && my_par == cur && my_tok == target;
    const unsigned b = __ballot_sync(0xffffffffu, match);
    if (!b) break;
    cur = __ffs(b) - 1;
    path[++d] = cur;
  }
  if (lane != 0) return;
  int toks[kMaxWidth + 1];
  for (int k = 0; k < d; ++k) toks[k] = tree->tok[path[k + 1]];
  toks[d] = pred[path[d]];
  const uint32_t L = ctl->committed_len;
  const uint32_t n_ctx = ctl->ctx_len;
  const uint32_t n_gen = ctl->n_generated;
  const uint32_t max_new = ctl->max_new;
  int e = d + 1;
  if ((uint32_t)e > max_new - n_gen) e = (int)(max_new - n_gen);
  bool hit_eos = false;
  if (eos >= 0) {
    for (int k = 0; k < e; ++k)
      if (toks[k] == eos) {
        e = k + 1;
        hit_eos = true;
        break;
      }
  }
  for (int k = 0; k < e; ++k) {
    ctx[n_ctx + k] = toks[k];
    wtok[wslot * kMaxWidth + k] = toks[k];
  }
  rec->valid = 1;
  rec->L_old = (int)L;
  rec->n_commit = e;
  rec->n_path = d + 1;
  for (int k = 0; k <= d; ++k) rec->path[k] = path[k];
  uint32_t nf = flags;
  const uint32_t nL = L + (uint32_t)e, nctx = n_ctx + (uint32_t)e, ngen = n_gen + (uint32_t)e;
  if (ngen >= max_new || hit_eos) nf |= FLAG_TERMINATED;
  else if (nL + (uint32_t)max_width > (uint32_t)kv_cap || nctx + kMaxCont + 1 > (uint32_t)ctx_cap) nf |= FLAG_ERR_CAPACITY;
  ctl->committed_len = nL;
  ctl->ctx_len = nctx;
  ctl->n_generated = ngen;
  ctl->root_tok = toks[e - 1];
  ctl->step_idx += 1;
  StepStats st;
  st.n_accepted_drafts = (uint16_t)d;
  st.best_match_len = (uint16_t)tree->best_len;
  st.n_nodes = (uint16_t)n_valid;
  st.n_emitted = (uint16_t)e;
  st.t_lo = globaltimer_lo();
  wstats[wslot] = st;
  __threadfence();
  ctl->flags = nf;
}

// Grid (layers * kv heads); each thread owns a set of dimensions and copies path rows in
// ascending order (path[j] >= j, so no source is overwritten before it is read).
__global__ void k_compact(const AcceptRec* __restrict__ rec, float* kc, float* vc, int Hkv, int kv_cap, int D) {
  griddep_enter();
  if (!rec->valid) return;
  const int n = rec->n_commit;
  const int L = rec->L_old;
  const size_t base = (size_t)blockIdx.x * kv_cap * D;  // (layer, kv head) block
  for (int j = 1; j < n; ++j) {
    const int src = rec->path[j];
    if (src == j) continue;
    const size_t so = base + (size_t)(L + src) * D, dof = base + (size_t)(L + j) * D;
    for (int dd = threadIdx.x; dd < D; dd += blockDim.x) {
      kc[dof + dd] = kc[so + dd];
      vc[dof + dd] = vc[so + dd];
    }
  }
}

// ------------------------------------------------------------------------------ drafter

constexpr int kDraftThreads = 512;
constexpr int kCand = 16;

__device__ __forceinline__ int block_excl_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  int pre = 0, tot = 0;
  for (int w = 0; w < kDraftThreads / 32; ++w) {
    if (w < warp) pre += s_warp[w];
    tot += s_warp[w];
  }
  *total = tot;
  return pre + x - v;
}

// One CTA of kDraftThreads.  Writes the full-width tree (kMaxWidth nodes) in best-first order:
// the first N nodes of it are the tree of width N.
// The scan covers the session memory (mem[0 .. *mem_len), earlier outputs each preceded by the
// separator -1, which equals no token) and then the context: scan position v < m is memory
// entry v, v >= m context position v - m.  A memory match stops at a separator, a memory
// continuation ends before the next one, and a higher scan position is the more recent.
__global__ void __launch_bounds__(kDraftThreads)
    k_draft(SpecCtl* ctl, const AcceptRec* __restrict__ rec, const int32_t* __restrict__ ctx,
            const int32_t* __restrict__ mem, const int* __restrict__ mem_len, TreeState* tree, int force) {
  griddep_enter();
  if (!force && (!rec->valid || (ctl->flags & FLAG_ERR_MASK))) return;
  extern __shared__ uint8_t s_ell[];  // match length per scan position
  __shared__ int s_suf[kMaxCont];
  __shared__ int s_warp[kDraftThreads / 32];
  __shared__ int s_cand[kCand];
  __shared__ int s_cont[kCand][kMaxCont];
  __shared__ int s_len[kCand], s_w[kCand];
  __shared__ int s_new[kCand][kMaxCont], s_score[kCand][kMaxCont], s_rep[kCand][kMaxCont], s_rank[kCand][kMaxCont];
  __shared__ int s_nnew;
  const int n = (int)ctl->ctx_len;
  const int m = mem_len != nullptr ? *mem_len : 0;
  const int tid = threadIdx.x;
  // past the context's start the suffix holds -2, which neither a token nor a separator equals
  if (tid < kMaxCont) s_suf[tid] = (n - 1 - tid >= 0) ? ctx[n - 1 - tid] : -2;
  if (tid < kCand) s_cand[tid] = -1;
  __syncthreads();
  // 1) match lengths over the scan positions [0, m + n - 2], each thread a descending segment
  const int P = m + n - 1;
  const int seg = (P + kDraftThreads - 1) / kDraftThreads;
  const int hi = P - 1 - tid * seg;  // highest position of this thread's segment
  const int lo = max(0, P - (tid + 1) * seg);
  int cnt[kMaxCont + 1];
#pragma unroll
  for (int l = 0; l <= kMaxCont; ++l) cnt[l] = 0;
  for (int v = hi; v >= lo; --v) {
    int l = 0;
    if (v >= m) {
      const int p = v - m;
      while (l < kMaxCont && p - l >= 0 && ctx[p - l] == s_suf[l]) ++l;
    } else {
      while (l < kMaxCont && v - l >= 0 && mem[v - l] == s_suf[l]) ++l;
    }
    s_ell[v] = (uint8_t)l;
    cnt[l] += 1;
  }
  // 2) rank of every matched position inside its class (descending position)
  int pre[kMaxCont + 1], tot[kMaxCont + 1];
  pre[0] = tot[0] = 0;
#pragma unroll
  for (int l = 1; l <= kMaxCont; ++l) pre[l] = block_excl_scan(cnt[l], s_warp, &tot[l]);
  int off[kMaxCont + 2];
  off[kMaxCont + 1] = 0;
#pragma unroll
  for (int l = kMaxCont; l >= 1; --l) off[l] = off[l + 1] + tot[l];
  const int n_cand = min(kCand, off[1]);
  {
    int run[kMaxCont + 1];
#pragma unroll
    for (int l = 0; l <= kMaxCont; ++l) run[l] = 0;
    for (int p = hi; p >= lo; --p) {
      const int l = s_ell[p];
      if (l == 0) continue;
      const int slot = off[l + 1] + pre[l] + run[l];
      run[l] += 1;
      if (slot < kCand) s_cand[slot] = p;
    }
  }
  __syncthreads();
  // 3) continuations of the candidates
  if (tid < kCand) {
    const int v = s_cand[tid];
    const bool on = tid < n_cand && v >= 0;
    int len = 0;
    if (on && v >= m) {
      const int p = v - m;
      len = min(kMaxCont, n - 1 - p);
      for (int k = 0; k < kMaxCont; ++k) s_cont[tid][k] = k < len ? ctx[p + 1 + k] : -1;
    } else {
      for (int k = 0; k < kMaxCont; ++k) {
        const int t = (on && v + 1 + k < m && len == k) ? mem[v + 1 + k] : -1;
        if (t >= 0) ++len;
        s_cont[tid][k] = k < len ? t : -1;
      }
    }
    s_len[tid] = len;
    s_w[tid] = on ? (int)s_ell[v] : 0;
  }
  __syncthreads();
  // 4) trie nodes = distinct prefixes; thread (i, L) for i < 16, L = 1..8
  const int ci = tid >> 3, cl = (tid & 7) + 1;
  if (tid < kCand * kMaxCont) {
    int rep = -1, score = 0;
    if (cl <= s_len[ci]) {
      for (int j = 0; j < kCand; ++j) {
        if (s_len[j] < cl) continue;
        bool eq = true;
        for (int k = 0; k < cl; ++k) eq = eq && (s_cont[j][k] == s_cont[ci][k]);
        if (!eq) continue;
        if (rep < 0) rep = j;
        score += s_w[j];
      }
    }
    s_rep[ci][cl - 1] = rep;
    s_new[ci][cl - 1] = (rep == ci) ? 1 : 0;
    s_score[ci][cl - 1] = score;
  }
  __syncthreads();
  if (tid < kCand * kMaxCont) {
    int rank = 0;
    if (s_new[ci][cl - 1]) {
      const int sc = s_score[ci][cl - 1];
      for (int j = 0; j < kCand; ++j)
        for (int k = 0; k < kMaxCont; ++k) {
          if (!s_new[j][k]) continue;
          const int sj = s_score[j][k], lj = k + 1;
          const bool better = sj > sc || (sj == sc && (lj < cl || (lj == cl && j < ci)));
          rank += better ? 1 : 0;
        }
    }
    s_rank[ci][cl - 1] = rank;
  }
  if (tid == 0) {
    int nn = 0;
    for (int j = 0; j < kCand; ++j)
      for (int k = 0; k < kMaxCont; ++k) nn += s_new[j][k];
    s_nnew = nn;
  }
  __syncthreads();
  const int n_valid = 1 + min(kMaxWidth - 1, s_nnew);
  if (tid < kMaxWidth) {  // default: padding nodes
    tree->tok[tid] = tid == 0 ? ctx[n - 1] : 0;
    tree->parent[tid] = tid == 0 ? -1 : 0;
    tree->depth[tid] = tid == 0 ? 0 : 1;
  }
  __syncthreads();
  if (tid < kCand * kMaxCont && s_new[ci][cl - 1]) {
    const int rank = s_rank[ci][cl - 1];
    if (rank < kMaxWidth - 1) {
      const int o = rank + 1;
      int par = 0;
      if (cl > 1) par = s_rank[s_rep[ci][cl - 2]][cl - 2] + 1;
      tree->tok[o] = s_cont[ci][cl - 1];
      tree->parent[o] = par;
      tree->depth[o] = cl;
    }
  }
  if (tid == 0) {
    tree->n_valid = n_valid;
    tree->best_len = n_cand > 0 ? (int)s_ell[s_cand[0]] : 0;
    ctl->n_valid = (uint32_t)n_valid;
  }
}

// Prefill: the next `len` prompt tokens ctx[L_c .. L_c+len) as a chain.
__global__ void k_chain_tree(const SpecCtl* ctl, const int32_t* __restrict__ ctx, TreeState* tree, int len) {
  griddep_enter();
  const int i = threadIdx.x;
  const int L = (int)ctl->committed_len;
  if (i < kMaxWidth) {
    tree->tok[i] = i < len ? ctx[L + i] : 0;
    tree->parent[i] = i == 0 ? -1 : (i < len ? i - 1 : 0);
    tree->depth[i] = i < len ? i : 1;
  }
  if (i == 0) {
    tree->n_valid = len;
    tree->best_len = 0;
  }
}

__global__ void k_commit_chain(SpecCtl* ctl, int len) {
  griddep_enter();
  if (threadIdx.x == 0 && !(ctl->flags & FLAG_ERR_MASK)) ctl->committed_len += (uint32_t)len;
}

cudaError_t launch_accept(const DecoderBufs& b, int N, int window_slot, cudaStream_t st) {
  return launch_pdl(k_accept, dim3(1), dim3(32), 0, st, b.ctl, (const TreeState*)b.tree, (const int32_t*)b.pred, N,
                    b.rec, b.ctx, b.ctx_cap, b.kv_cap, kMaxWidth, b.wstats, b.wtok, window_slot, b.eos_id);
}

cudaError_t launch_compact(const DecoderBufs& b, const ModelDims& m, cudaStream_t st) {
  return launch_pdl(k_compact, dim3(m.n_layers * m.Hkv), dim3(128), 0, st, (const AcceptRec*)b.rec, b.kcache,
                    b.vcache, m.Hkv, b.kv_cap, m.D);
}

cudaError_t launch_draft(const DecoderBufs& b, int force, cudaStream_t st) {
  return launch_pdl(k_draft, dim3(1), dim3(kDraftThreads), (size_t)b.ctx_cap + b.mem_cap, st, b.ctl,
                    (const AcceptRec*)b.rec, (const int32_t*)b.ctx, (const int32_t*)b.mem, (const int*)b.mem_len,
                    b.tree, force);
}

cudaError_t draft_configure(int scan_cap) {
  // the attribute is per kernel, shared by every session: only ever raised
  static int configured = 0;
  if (scan_cap <= configured) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(k_draft, cudaFuncAttributeMaxDynamicSharedMemorySize, scan_cap);
  if (e == cudaSuccess) configured = scan_cap;
  return e;
}

cudaError_t launch_chain_tree(const DecoderBufs& b, int start, int len, cudaStream_t st) {
  (void)start;
  return launch_pdl(k_chain_tree, dim3(1), dim3(32), 0, st, (const SpecCtl*)b.ctl, (const int32_t*)b.ctx, b.tree,
                    len);
}

cudaError_t launch_commit_chain(const DecoderBufs& b, int len, cudaStream_t st) {
  return launch_pdl(k_commit_chain, dim3(1), dim3(32), 0, st, b.ctl, len);
}

}  // namespace w4a8
