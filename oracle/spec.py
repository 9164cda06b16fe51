"""Tree verification, greedy acceptance, KV compaction, the suffix n-gram drafter
and the speculative decoding loop, step by step.

"GPU-Resident Speculative Decoding ...", Design > GPU-Resident Speculation Loop:
a step processes N tree nodes (node 0 = the token produced by the previous
step, nodes 1..N-1 the draft tree); every node attends to the committed cache
and to its ancestors; acceptance walks the tree from the root, following the
child whose token equals the greedy prediction of its parent; the step commits
the accepted drafts plus the token predicted after the last of them (1..N
tokens, at most 9 because a candidate is extended by at most 8 tokens);
compaction moves the accepted path's keys and values into place; the drafter
writes the next tree.
"Exact Speculative And Assisted Decoding ...", section 4 (greedy: accept iff the
proposal equals the target argmax; bonus token after a full acceptance) and
section 7 (commit/rollback is a move of the logical length, no zeroing).
Design > Draft-Free Drafting From Web Context: match length of every context
position with the current suffix at orders up to 8, selection of the best
positions, a weighted trie of their continuations, emission of the most
probable prefix-closed node set.

Readings where the pages leave a step open:
* matched positions p in [0, n-2]; l(p) = largest l <= 8 with
  c[p-l+1..p] == c[n-l..n-1]; candidates are the 16 best by (l desc, p desc)
  among l >= 1; a candidate continues with c[p+1 .. min(p+8, n-1)] with weight
  l; trie score = sum of weights through a node; nodes are taken best-first by
  (score desc, depth asc, insertion order asc); unused nodes are invalid
  (token 0, parent 0).
* among children with the predicted token, the lowest node index is followed.
* a step stops emitting at ``max_new`` tokens in total, or after an ``eos``.
"""
from __future__ import annotations

import heapq

import numpy as np

from .model import Model, argmax_lowest, attend, kv_head_of

MAX_ORDER = 8
N_CAND = 16
MAX_CONT = 8


def tree_depths(parent) -> np.ndarray:
    n = len(parent)
    depth = np.zeros(n, dtype=np.int32)
    for i in range(1, n):
        assert 0 <= parent[i] < i
        depth[i] = depth[parent[i]] + 1
    return depth


def ancestors_or_self(parent, i) -> list:
    """Nodes on the path root..i, root first."""
    path = []
    while i >= 0:
        path.append(int(i))
        i = int(parent[i]) if i > 0 else -1
    return path[::-1]


def tree_visible(L_c: int, parent, i: int) -> list:
    """Cache slots node i sees in a verification step: [0, L_c), then the slots L_c + a of
    its root path (a node's K/V sits at slot L_c + its index)."""
    return list(range(L_c)) + [L_c + a for a in ancestors_or_self(parent, i)]


def tree_attention(qs: np.ndarray, K: np.ndarray, V: np.ndarray, L_c: int, parent) -> np.ndarray:
    """Attention of every tree node over the slots it sees (Design > GPU-Resident
    Speculation Loop: each node attends to the committed cache and to its ancestors).
    qs: [n][Hq][d] queries already multiplied by 1/sqrt(d); K, V: [Hkv][slots][d].
    Returns fp64 [n][Hq][d]: softmax(qs . k) v over the visible slots, query head h
    reading KV head h // (Hq / Hkv)."""
    n, Hq, d = qs.shape
    Hkv = K.shape[0]
    out = np.zeros((n, Hq, d))
    for i in range(n):
        vis = np.asarray(tree_visible(L_c, parent, i), dtype=np.int64)
        for h in range(Hq):
            kh = kv_head_of(h, Hq, Hkv)
            # attend divides the scores by sqrt(d): undo the factor the queries carry
            out[i, h] = attend(np.asarray(qs[i, h], dtype=np.float64) * np.sqrt(d), K[kh, vis], V[kh, vis])
    return out


def tree_verify(model: Model, L_c: int, tok, parent) -> np.ndarray:
    """Logits of every tree node; node i sits at logical position L_c + depth(i), writes
    its K/V to slot L_c + i and sees cache slots [0, L_c) then its root path."""
    depth = tree_depths(parent)
    n = len(tok)
    vis = [tree_visible(L_c, parent, i) for i in range(n)]
    return model.forward(list(tok), [L_c + int(depth[i]) for i in range(n)],
                         [L_c + i for i in range(n)], vis)


def accept(tok, parent, pred, n_valid: int):
    """Greedy tree acceptance.  Returns (path of node indices from 0, emitted tokens)."""
    path = [0]
    cur = 0
    while True:
        nxt = None
        for j in range(1, n_valid):
            if parent[j] == cur and tok[j] == pred[cur]:
                nxt = j
                break
        if nxt is None:
            break
        path.append(nxt)
        cur = nxt
    emitted = [int(tok[j]) for j in path[1:]] + [int(pred[path[-1]])]
    return path, emitted


def compact(model: Model, L_c: int, path) -> None:
    """Move the K/V of accepted node path[j] (slot L_c + path[j]) to slot L_c + j, j ascending."""
    for l in range(model.shape.n_layers):
        for j in range(1, len(path)):
            model.K[l][:, L_c + j] = model.K[l][:, L_c + path[j]]
            model.V[l][:, L_c + j] = model.V[l][:, L_c + path[j]]


def match_lengths(ctx, max_order: int = MAX_ORDER) -> np.ndarray:
    """l(p) for p in [0, n-2]: length of the match ending at p with the context suffix."""
    c = [int(t) for t in ctx]
    n = len(c)
    out = np.zeros(max(n - 1, 0), dtype=np.int32)
    for p in range(n - 1):
        l = 0
        while l < max_order and p - l >= 0 and c[p - l] == c[n - 1 - l]:
            l += 1
        out[p] = l
    return out


SEP = -1  # separates the earlier outputs held in a session memory (equal to no token)


def memory_array(segments, cap: int = 1 << 15):
    """The session memory of Design > Draft-Free Drafting From Web Context (the drafter's scan
    also covers a buffer of the model's outputs from earlier requests), as one token array:
    every earlier output preceded by SEP, oldest first, keeping at most ``cap`` entries (whole
    outputs are dropped from the oldest; an output longer than the memory keeps its last
    cap - 1 tokens)."""
    mem = []
    for seg in segments:
        seg = [int(t) for t in seg]
        if len(seg) + 1 > cap:
            seg = seg[len(seg) - (cap - 1):]
        while mem and len(mem) + len(seg) + 1 > cap:
            nxt = mem.index(SEP, 1) if SEP in mem[1:] else len(mem)
            mem = mem[nxt:]
        mem += [SEP] + seg
    return mem


def match_lengths_with_memory(mem, ctx, max_order: int = MAX_ORDER) -> np.ndarray:
    """l(v) over the scan positions v of the sequence mem + ctx (every memory position, then the
    context positions but its last): the length of the run of tokens ending at v that equals the
    context suffix, within the memory (a SEP ends it) or within the context."""
    m = len(mem)
    c = [int(t) for t in ctx]
    n = len(c)
    out = np.zeros(m + max(n - 1, 0), dtype=np.int32)
    for v in range(m):
        l = 0
        while l < max_order and v - l >= 0 and l < n and mem[v - l] == c[n - 1 - l]:
            l += 1
        out[v] = l
    out[m:] = match_lengths(c, max_order)
    return out


def draft(ctx, N: int, n_cand: int = N_CAND, max_cont: int = MAX_CONT, memory=()):
    """Next tree of N nodes from context ``ctx`` (whose last token is the root) and an optional
    session memory (``memory_array``), scanned as if it preceded the context: a memory match
    continues with the tokens after it up to the next SEP, and among equal match lengths a
    context position is more recent than any memory position.

    Returns (tok int32[N], parent int32[N] with parent[0] = -1, n_valid, best_match_len)."""
    c = [int(t) for t in ctx]
    n = len(c)
    mem = [int(t) for t in memory]
    m = len(mem)
    ell = match_lengths_with_memory(mem, c)
    cand = sorted((v for v in range(len(ell)) if ell[v] >= 1), key=lambda v: (-int(ell[v]), -v))[:n_cand]
    best = int(ell[cand[0]]) if cand else 0

    def continuation(v):
        if v >= m:
            p = v - m
            return c[p + 1: min(p + max_cont, n - 1) + 1]
        out = []
        for t in mem[v + 1: v + 1 + max_cont]:
            if t == SEP:
                break
            out.append(t)
        return out

    # weighted trie; node 0 is the root token
    node_tok, node_par, node_dep, node_score = [c[-1]], [-1], [0], [0]
    children = {}
    for p in cand:
        w = int(ell[p])
        cur = 0
        for t in continuation(p):
            key = (cur, t)
            if key not in children:
                children[key] = len(node_tok)
                node_tok.append(t)
                node_par.append(cur)
                node_dep.append(node_dep[cur] + 1)
                node_score.append(0)
            cur = children[key]
            node_score[cur] += w
    kids = {}
    for (par, _t), nd in children.items():
        kids.setdefault(par, []).append(nd)
    # best-first expansion: (score desc, depth asc, insertion order asc)
    heap = [(-node_score[nd], node_dep[nd], nd) for nd in kids.get(0, [])]
    heapq.heapify(heap)
    picked = []
    while heap and len(picked) < N - 1:
        _, _, nd = heapq.heappop(heap)
        picked.append(nd)
        for ch in kids.get(nd, []):
            heapq.heappush(heap, (-node_score[ch], node_dep[ch], ch))
    out_idx = {0: 0}
    tok = np.zeros(N, dtype=np.int32)
    parent = np.zeros(N, dtype=np.int32)
    tok[0], parent[0] = c[-1], -1
    for i, nd in enumerate(picked):
        out_idx[nd] = i + 1
        tok[i + 1] = node_tok[nd]
        parent[i + 1] = out_idx[node_par[nd]]
    return tok, parent, 1 + len(picked), best


def spec_decode(weights, prompt, max_new: int, widths, eos: int = -1, kv_cap: int | None = None,
                record=None, memory=()):
    """Speculative greedy decoding.  ``widths`` is an int or a callable step -> N; ``memory`` a
    session memory (``memory_array``) the drafter scans besides the context.

    Returns (tokens, stats) with stats = list of (n_accepted_drafts, best_match_len, n_valid)."""
    prompt = [int(t) for t in prompt]
    n = len(prompt)
    wfun = widths if callable(widths) else (lambda _s, _w=int(widths): _w)
    nmax = 32
    m = Model(weights, kv_cap or (n + max_new + nmax + 1))
    if n > 1:
        m.prefill(prompt[:-1], head=False)
    L_c = n - 1
    ctx = list(prompt)
    out, stats = [], []
    step = 0
    while len(out) < max_new:
        N = int(wfun(step))
        tok, parent, n_valid, best = draft(ctx, N, memory=memory)
        logits = tree_verify(m, L_c, tok, parent)
        pred = [argmax_lowest(logits[i]) for i in range(N)]
        path, emitted = accept(tok, parent, pred, n_valid)
        e = min(len(emitted), max_new - len(out))
        if eos >= 0 and eos in emitted[:e]:
            e = emitted.index(eos) + 1
        emitted = emitted[:e]
        compact(m, L_c, path[:e])
        if record is not None:
            record.append(dict(N=N, L_c=L_c, tok=tok.copy(), parent=parent.copy(), n_valid=n_valid,
                               logits=logits, pred=pred, path=path, emitted=emitted))
        L_c += e
        ctx += emitted
        out += emitted
        stats.append((len(path) - 1, best, n_valid))
        step += 1
        if eos >= 0 and emitted and emitted[-1] == eos:
            break
    return out, stats
