"""Pins of the oracle's acceptance, compaction, drafter and speculative loop (CPU)."""
import itertools

import numpy as np
import pytest

import synth
from oracle import model as OM
from oracle import spec as OS


def _all_root_paths(parent, n_valid):
    kids = {i: [j for j in range(1, n_valid) if parent[j] == i] for i in range(n_valid)}
    out = []
    def rec(p):
        out.append(list(p))
        for c in kids[p[-1]]:
            rec(p + [c])
    rec([0])
    return out


@pytest.mark.parametrize("seed", range(40))
def test_accept_is_longest_matching_path(seed):
    # In a real verification the prediction after a node depends only on the tokens of
    # its root path, so duplicated siblings predict alike; model that with a hash of the
    # path's tokens.  The walk then finds a longest root path whose every edge matches.
    rng = np.random.default_rng(seed)
    N = int(rng.integers(1, 17))
    n_valid = int(rng.integers(1, N + 1))
    V = 3                                                   # tiny vocab: many matches and duplicates
    tok, parent = synth.random_tree(rng, N, V, n_valid=n_valid)
    table = {}
    def pred_of(i):
        key = tuple(int(tok[j]) for j in OS.ancestors_or_self(parent, i))
        if key not in table:
            table[key] = int(rng.integers(0, V))
        return table[key]
    pred = [pred_of(i) for i in range(N)]
    path, emitted = OS.accept(tok, parent, pred, n_valid)
    ok = [p for p in _all_root_paths(parent, n_valid)
          if all(tok[p[i + 1]] == pred[p[i]] for i in range(len(p) - 1))]
    assert len(path) == max(len(p) for p in ok)
    assert path in ok
    assert emitted == [int(tok[j]) for j in path[1:]] + [pred[path[-1]]]
    assert 1 <= len(emitted) <= n_valid


@pytest.mark.parametrize("seed", range(20))
def test_accept_walk_rule_arbitrary_predictions(seed):
    # with arbitrary predictions: every step takes the lowest-index matching child, and
    # the walk stops only where no valid child matches
    rng = np.random.default_rng(1000 + seed)
    N = int(rng.integers(1, 17))
    n_valid = int(rng.integers(1, N + 1))
    tok, parent = synth.random_tree(rng, N, 3, n_valid=n_valid)
    pred = rng.integers(0, 3, size=N).tolist()
    path, _ = OS.accept(tok, parent, pred, n_valid)
    for a, b in zip(path, path[1:]):
        match = [j for j in range(1, n_valid) if parent[j] == a and tok[j] == pred[a]]
        assert b == min(match)
    assert not [j for j in range(1, n_valid) if parent[j] == path[-1] and tok[j] == pred[path[-1]]]


def test_accept_chain_is_longest_matching_prefix():
    # a chain tree reduces to the linear rule: accept drafts while they equal the argmax
    tok = [7, 1, 2, 3, 4]
    parent = [-1, 0, 1, 2, 3]
    pred = [1, 2, 9, 4, 5]
    path, emitted = OS.accept(tok, parent, pred, 5)
    assert path == [0, 1, 2] and emitted == [1, 2, 9]
    path, emitted = OS.accept(tok, parent, [1, 2, 3, 4, 6], 5)
    assert path == [0, 1, 2, 3, 4] and emitted == [1, 2, 3, 4, 6]     # full accept + bonus


def test_compact_moves_path_rows():
    w = OM.build_weights(synth.ModelShape("c", 1, 64, 4, 2, 16, 64, 64, 64, False), 1)
    m = OM.Model(w, 12)
    for l in range(1):
        m.K[l][:] = np.arange(12, dtype=np.float32)[None, :, None]
        m.V[l][:] = -np.arange(12, dtype=np.float32)[None, :, None]
    OS.compact(m, 4, [0, 2, 5, 7])
    assert m.K[0][0, :, 0].tolist() == [0, 1, 2, 3, 4, 6, 9, 11, 8, 9, 10, 11]
    assert m.V[0][1, :, 3].tolist() == [-v for v in [0, 1, 2, 3, 4, 6, 9, 11, 8, 9, 10, 11]]


def _brute_match(ctx, p, max_order=8):
    best = 0
    for l in range(1, max_order + 1):
        if p - l + 1 < 0:
            break
        if ctx[p - l + 1:p + 1] == ctx[len(ctx) - l:]:
            best = l
    return best


@pytest.mark.parametrize("seed", range(10))
def test_match_lengths_brute_force(seed):
    rng = np.random.default_rng(seed)
    ctx = rng.integers(0, 3, size=int(rng.integers(2, 60))).tolist()
    ell = OS.match_lengths(ctx)
    assert ell.tolist() == [_brute_match(ctx, p) for p in range(len(ctx) - 1)]


def test_draft_single_candidate_is_prompt_lookup_chain():
    # one earlier occurrence of the last token: the tree is the chain of its continuation
    ctx = [10, 11, 12, 13, 14, 15, 16, 17, 18, 19, 20, 21, 10]
    tok, parent, n_valid, best = OS.draft(ctx, 8)
    assert best == 1 and n_valid == 8
    assert tok.tolist() == [10, 11, 12, 13, 14, 15, 16, 17]
    assert parent.tolist() == [-1, 0, 1, 2, 3, 4, 5, 6]
    # continuation stops at 8 tokens and at the end of the context
    tok, parent, n_valid, _ = OS.draft(ctx, 16)
    assert n_valid == 9 and tok[1:9].tolist() == [11, 12, 13, 14, 15, 16, 17, 18]
    assert tok[9:].tolist() == [0] * 7 and parent[9:].tolist() == [0] * 7


def test_draft_no_match():
    tok, parent, n_valid, best = OS.draft([1, 2, 3, 4], 4)
    assert n_valid == 1 and best == 0 and tok[0] == 4


def test_draft_scores_prefer_longer_matches():
    # suffix "5 6" occurs twice: after "1 5 6" continues 7, after "2 5 6"... the longer match wins first
    ctx = [9, 5, 6, 7, 1, 3, 5, 6, 8, 2, 9, 5, 6]
    ell = OS.match_lengths(ctx)
    assert ell[2] == 3 and ell[7] == 2
    tok, parent, n_valid, best = OS.draft(ctx, 3)
    assert best == 3
    assert tok[1] == 7                     # continuation of the order-3 match has the larger score


@pytest.mark.parametrize("seed", range(20))
def test_draft_tree_is_prefix_closed_and_ordered(seed):
    rng = np.random.default_rng(seed)
    motifs = rng.integers(0, 20, size=(3, 6))
    ctx = np.concatenate([motifs[i] for i in rng.integers(0, 3, size=12)]).tolist()
    N = int(rng.integers(2, 17))
    tok, parent, n_valid, best = OS.draft(ctx, N)
    assert tok[0] == ctx[-1] and parent[0] == -1
    for i in range(1, n_valid):
        assert 0 <= parent[i] < i
    # siblings are distinct tokens
    for i in range(n_valid):
        sib = [tok[j] for j in range(1, n_valid) if parent[j] == i]
        assert len(sib) == len(set(sib))
    # every root path of the tree is a continuation present in the context after a match
    depth = OS.tree_depths(parent)
    assert depth[:n_valid].max() <= 8


def _weights():
    return OM.build_weights(synth.TINY, 1000)


@pytest.fixture(scope="module")
def tiny():
    w = _weights()
    prompt = synth.motif_prompt(1001, 64, 4, 16, 0.1, synth.TINY.vocab)
    greedy, _ = OM.greedy_decode(w, prompt, 32)
    return w, prompt, greedy


@pytest.mark.parametrize("N", [1, 2, 4, 8, 16])
def test_speculative_equals_greedy(tiny, N):
    w, prompt, greedy = tiny
    out, stats = OS.spec_decode(w, prompt, 32, N)
    assert out == greedy
    for d, _best, n_valid in stats:
        assert 0 <= d <= min(n_valid - 1, 8)


def test_speculative_equals_greedy_with_varying_width(tiny):
    w, prompt, greedy = tiny
    widths = [1, 8, 2, 16, 4, 1, 3]
    out, _ = OS.spec_decode(w, prompt, 32, lambda s: widths[s % len(widths)])
    assert out == greedy


def test_accepted_prefix_kv_equals_sequential_kv(tiny):
    w, prompt, greedy = tiny
    n = len(prompt)
    rec = []
    OS.spec_decode(w, prompt, 12, 8, record=rec)
    # rebuild the spec model's cache state by replaying, then compare with a plain prefill
    m = OM.Model(w, n + 64)
    m.prefill(list(prompt[:-1]))
    L_c = n - 1
    for r in rec:
        OS.tree_verify(m, L_c, r["tok"], r["parent"])
        OS.compact(m, L_c, r["path"][:len(r["emitted"])])
        L_c += len(r["emitted"])
    seq = OM.Model(w, n + 64)
    seq.prefill(list(prompt) + greedy[:L_c - n])
    for l in range(synth.TINY.n_layers):
        assert np.array_equal(m.K[l][:, :L_c], seq.K[l][:, :L_c])
        assert np.array_equal(m.V[l][:, :L_c], seq.V[l][:, :L_c])


def test_max_new_truncates_and_eos_stops(tiny):
    w, prompt, greedy = tiny
    out, _ = OS.spec_decode(w, prompt, 5, 16)
    assert out == greedy[:5]
    eos = greedy[3]
    out, _ = OS.spec_decode(w, prompt, 32, 8, eos=eos)
    assert out == greedy[:greedy.index(eos) + 1]


# ------------------------------------------------------------------ tree attention pins

def _attn_case(seed, n_heads=4, n_kv=2, d=8, L=5, n=6):
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((n_kv, L + n, d))
    V = rng.standard_normal((n_kv, L + n, d))
    qs = rng.standard_normal((n, n_heads, d)) / np.sqrt(d)
    return qs, K, V


def test_tree_attention_chain_is_causal_attention():
    # a chain's node i sees every slot up to L + i: plain causal softmax attention, written out
    qs, K, V = _attn_case(1)
    L, n = 5, 6
    out = OS.tree_attention(qs, K, V, L, [-1] + list(range(n - 1)))
    for i in range(n):
        for h in range(4):
            kh = h // 2
            sc = K[kh, :L + i + 1] @ qs[i, h]
            w = np.exp(sc - sc.max())
            assert np.allclose(out[i, h], (w / w.sum()) @ V[kh, :L + i + 1], rtol=1e-12, atol=1e-12)


def test_tree_attention_star_sees_root_and_itself():
    # every node a child of the root: node i sees [0, L), slot L (root) and slot L + i
    qs, K, V = _attn_case(2)
    L, n = 5, 6
    out = OS.tree_attention(qs, K, V, L, [-1] + [0] * (n - 1))
    for i in range(1, n):
        vis = [0, 1, 2, 3, 4, L, L + i]
        for h in range(4):
            kh = h // 2
            sc = K[kh, vis] @ qs[i, h]
            w = np.exp(sc - sc.max())
            assert np.allclose(out[i, h], (w / w.sum()) @ V[kh, vis], rtol=1e-12, atol=1e-12)


def test_tree_attention_ignores_slots_off_the_path():
    # tree 0 -> 1 -> 3, 0 -> 2: node 3 must not see node 2's slot; node 2 must not see 1 or 3
    qs, K, V = _attn_case(3, n=4)
    L = 5
    parent = [-1, 0, 0, 1]
    base = OS.tree_attention(qs, K, V, L, parent)
    K2, V2 = K.copy(), V.copy()
    K2[:, L + 2] += 5.0
    V2[:, L + 2] -= 3.0
    moved = OS.tree_attention(qs, K2, V2, L, parent)
    assert np.array_equal(base[3], moved[3]) and np.array_equal(base[1], moved[1])
    assert not np.allclose(base[2], moved[2])
    K3 = K.copy()
    K3[:, L + 1] += 5.0  # an ancestor of node 3: its output changes
    assert not np.allclose(OS.tree_attention(qs, K3, V, L, parent)[3], base[3])


def test_tree_attention_uses_the_grouped_kv_head():
    # V of KV head 1 zeroed: query heads 2, 3 (group of KV head 1) give zero, heads 0, 1 do not
    qs, K, V = _attn_case(4)
    V[1] = 0.0
    out = OS.tree_attention(qs, K, V, 5, [-1, 0, 1, 1, 0, 4])
    assert np.all(out[:, 2:] == 0.0)
    assert np.all(np.abs(out[:, :2]).sum(axis=-1) > 0)


# ---------------------------------------------------------------- drafter scoring pins
# Draft-Free Drafting From Web Context: candidates are weighted by a fixed function of
# their match length (read: w = l), at most 16 candidates are kept (most recent first
# among equal lengths), and trie nodes are taken best-first by (score desc, depth asc,
# insertion asc).  Each context below is built so that one plausible misreading picks a
# different first node; the match lengths it relies on are asserted first.

def test_draft_weight_is_match_length_not_count():
    X, Y, Z, A, B = 101, 102, 103, 104, 105
    ctx = [X, Y, Z, A, 7, Z, B, 8, Z, B, 9, X, Y, Z]
    ell = OS.match_lengths(ctx)
    assert ell[2] == 3 and ell[5] == 1 and ell[8] == 1
    assert sorted(int(v) for v in ell if v > 0) == [1, 1, 3]
    tok, parent, n_valid, best = OS.draft(ctx, 2)
    # w = l: A scores 3 against B's 1 + 1; a count (w = 1) would rank B (2) above A (1)
    assert best == 3 and tok[1] == A and parent[1] == 0
    # the whole order-3 continuation (score 3 at every depth) precedes B at depth 1 (score 2)
    tok, parent, n_valid, _ = OS.draft(ctx, 10)
    assert tok[1:10].tolist() == [A, 7, Z, B, 8, Z, B, 9, B]
    assert parent[1:10].tolist() == [0, 1, 2, 3, 4, 5, 6, 7, 0]


def test_draft_keeps_at_most_16_candidates_most_recent_first():
    R = 999
    follow = list(range(201, 217))                     # B1..B16 after the 16 most recent R
    ctx = [R, follow[-1], 5]                           # the 17th (oldest) R is also followed by B16
    for b in reversed(follow):
        ctx += [R, b, 6]
    ctx += [777, R]
    ell = OS.match_lengths(ctx)
    assert int((ell >= 1).sum()) == 17 and int(ell.max()) == 1
    tok, parent, n_valid, best = OS.draft(ctx, 2)
    # cap 16: B16 keeps score 1 and the most recent candidate's B1 comes first; without the
    # cap B16 would score 2
    assert best == 1 and tok[1] == follow[0]
    tok, _, _, _ = OS.draft(ctx, 16)
    assert tok[1:16].tolist() == follow[:15]          # equal scores: insertion (recency) order


def test_draft_ties_prefer_shallow_nodes_then_insertion():
    R, P, Q, S = 300, 301, 302, 303
    # two order-1 candidates: the most recent continues P Q, the older one S
    ctx = [R, S, 9, 9, 9, 9, 9, 9, 9, 9, R, P, Q, 8, 8, 8, 8, 8, 8, 8, 8, R]
    ell = OS.match_lengths(ctx)
    assert [p for p in range(len(ctx) - 1) if ell[p] >= 1] == [0, 10] and int(ell.max()) == 1
    tok, parent, n_valid, _ = OS.draft(ctx, 3)
    # P (score 1, depth 1, inserted first), then S (score 1, depth 1) before Q (score 1, depth 2)
    assert tok[1:3].tolist() == [P, S] and parent[1:3].tolist() == [0, 0]


def test_draft_score_outranks_depth():
    R, P, Q, S = 400, 401, 402, 403
    # an order-2 candidate continues P Q; an order-1 candidate continues S
    ctx = [7, R, P, Q, 5, 5, 5, 5, 5, 5, 5, 5, 6, R, S, 5, 5, 5, 5, 5, 5, 5, 5, 7, R]
    ell = OS.match_lengths(ctx)
    assert ell[1] == 2 and ell[13] == 1
    tok, parent, n_valid, best = OS.draft(ctx, 3)
    # Q (score 2, depth 2) before S (score 1, depth 1)
    assert best == 2 and tok[1:3].tolist() == [P, Q] and parent[1:3].tolist() == [0, 1]


# ------------------------------------------------------------------ session memory pins
# Draft-Free Drafting From Web Context: a memory region holds earlier outputs and the same scan
# searches it.  Reading: outputs are separated by SEP, a match or a continuation never crosses a
# SEP, and the memory counts as older than the context.

def test_memory_array_keeps_whole_recent_outputs():
    S = OS.SEP
    assert OS.memory_array([[1, 2], [3]]) == [S, 1, 2, S, 3]
    assert OS.memory_array([[1, 2, 3], [4, 5], [6]], cap=6) == [S, 4, 5, S, 6]   # oldest output dropped
    assert OS.memory_array([list(range(10))], cap=5) == [S, 6, 7, 8, 9]           # last cap - 1 tokens
    assert OS.memory_array([]) == []


def _brute_mem_ell(mem, ctx, v, max_order=8):
    seq = mem + ctx
    m = len(mem)
    lo = 0 if v < m else m                     # a match stays inside the memory or the context
    best = 0
    for l in range(1, max_order + 1):
        if v - l + 1 < lo or l > len(ctx):
            break
        if seq[v - l + 1:v + 1] == ctx[len(ctx) - l:]:
            best = l
    return best


@pytest.mark.parametrize("seed", range(10))
def test_memory_match_lengths_brute_force(seed):
    rng = np.random.default_rng(700 + seed)
    segs = [rng.integers(0, 3, size=int(rng.integers(1, 12))).tolist() for _ in range(int(rng.integers(0, 4)))]
    mem = OS.memory_array(segs)
    ctx = rng.integers(0, 3, size=int(rng.integers(2, 30))).tolist()
    ell = OS.match_lengths_with_memory(mem, ctx)
    assert ell.tolist() == [_brute_mem_ell(mem, ctx, v) for v in range(len(mem) + len(ctx) - 1)]


def test_memory_only_match_drafts_its_continuation_up_to_the_separator():
    mem = OS.memory_array([[50, 51, 52, 53], [60, 61]])
    tok, parent, n_valid, best = OS.draft([7, 8, 51], 8, memory=mem)
    assert best == 1 and n_valid == 3 and tok[1:3].tolist() == [52, 53]        # stops at the SEP before 60
    assert parent[1:3].tolist() == [0, 1]
    tok, _, n_valid, _ = OS.draft([7, 8, 51], 8)                                # no memory: nothing to draft
    assert n_valid == 1


def test_memory_match_does_not_cross_an_output_boundary():
    mem = OS.memory_array([[9], [5, 6]])                     # [SEP, 9, SEP, 5, 6]
    ell = OS.match_lengths_with_memory(mem, [1, 9, 5])
    assert ell[3] == 1                                       # 5 is preceded by SEP, not by 9


def test_context_is_more_recent_than_memory_at_equal_length():
    R = 40
    mem = OS.memory_array([[R, 41]])
    tok, _, _, best = OS.draft([R, 42, 3, R], 2, memory=mem)
    assert best == 1 and tok[1] == 42
    # a longer match in the memory outranks a shorter one in the context
    mem = OS.memory_array([[77, R, 41]])
    tok, _, _, best = OS.draft([R, 42, 3, 77, R], 2, memory=mem)
    assert best == 2 and tok[1] == 41
