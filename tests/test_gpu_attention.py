"""Tree attention through the C ABI (w4a8_session_attention) against its definition, and
the exactness invariants of the verification pass on the attention shapes of the
benchmark workload.

Parity: node i of a tree over committed length L sees cache slots [0, L) and the slots
L + a of its ancestors-or-self ("GPU-Resident Speculative Decoding ...", Design >
GPU-Resident Speculation Loop); its output for query head h is the softmax-weighted sum
of the values of KV head h // G.  The cache holds what the library's own prefill and one
verification pass wrote (read back with w4a8_session_copy_kv); the queries are seeded
random; the oracle evaluates the definition in fp64.  The kernel forms scores and value
sums on the tensor cores from f16 hi/lo splits of fp32 operands with fp32 accumulation
(about 2^-21 relative per product), so each output must lie within 2e-5 * max|V| of the
oracle.

Shapes (1 layer each, random init): head size 128 with 4 query heads per KV head and 8
KV heads (the grouping of the Llama-3-8B workload; with a 2048-slot cache every split CTA
takes two 64-position chunks), and head size 64 with 7 query heads per KV head (a node's
queries straddle two 16-row tiles).  Committed lengths cover a ragged chunk, a tree that
crosses a chunk boundary, a tree that starts a new chunk and a one-token context.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import synth
import synth.cuda as SC
import w4a8_verify_gb300 as W
from w4a8_verify_gb300 import models as WM
from oracle import spec as OS

pytestmark = pytest.mark.gpu

SEED = 1100
D128 = synth.ModelShape("d128-g4-kv8-1L", 1, 4096, 32, 8, 128, 1024, 1024, 1024, False)
D64G7 = synth.ModelShape("d64-g7-kv2-1L", 1, 896, 14, 2, 64, 1024, 1024, 1024, False)
KV_CAP = {D128.name: 2048, D64G7.name: 512}
ATOL_V = 2e-5


def _fill(shape, seed):
    def fill(kind, layer, out):
        if kind == W.T_EMBED:
            SC.dense_weight(shape, seed, synth.STREAM_EMBED, shape.vocab, shape.hidden, shape.vocab, shape.hidden, out)
        elif kind == W.T_LM_HEAD:
            SC.dense_weight(shape, seed, synth.STREAM_LM_HEAD, shape.vocab, shape.hidden, shape.vocab, shape.hidden,
                            out)
        else:
            rows, cols, rr, rc = synth.tensor_shape(shape, kind)
            SC.dense_weight(shape, seed, synth.layer_stream(layer, kind), rows, cols, rr, rc, out)
    return fill


_models = {}


def _model(shape):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if shape.name not in _models:
        W.lib()
        SC.lib()
        _models[shape.name] = WM.build_model(shape.n_layers, shape.hidden, shape.n_heads, shape.n_kv_heads,
                                             shape.head_dim, shape.ffn, shape.vocab, shape.tied,
                                             _fill(shape, SEED), shape.rms_eps, shape.rope_base)
    return _models[shape.name]


def _session(shape):
    return W.Session(_model(shape), KV_CAP[shape.name], KV_CAP[shape.name] + 64, 16, -1)


def _dev(a):
    return torch.as_tensor(np.asarray(a), dtype=torch.int32).cuda()


def _tree(kind, rng, n, vocab):
    if kind == "chain":
        return rng.integers(0, vocab, n), np.array([-1] + list(range(n - 1)))
    if kind == "star":
        return rng.integers(0, vocab, n), np.array([-1] + [0] * (n - 1))
    return synth.random_tree(rng, n, vocab)


CASES = [
    # (shape, committed length L, tree kind, nodes)
    (D128, 130, "random", 16),   # ragged chunk; split 0 takes chunks 0, 1
    (D128, 185, "chain", 16),    # the chain crosses position 192 (chunk boundary)
    (D128, 192, "random", 16),   # the tree starts chunk 3 (no cached slot in it)
    (D128, 300, "star", 16),     # five chunks over three split CTAs
    (D128, 250, "random", 11),
    (D128, 77, "random", 5),
    (D128, 140, "chain", 2),
    (D128, 1, "random", 16),     # one committed token
    (D128, 129, "random", 1),
    (D64G7, 130, "random", 16),  # 7 queries per node: nodes straddle 16-row tiles
    (D64G7, 191, "chain", 16),
    (D64G7, 64, "star", 9),
    (D64G7, 33, "random", 3),
]


@pytest.mark.parametrize("shape,L,kind,n", CASES, ids=lambda v: getattr(v, "name", str(v)))
def test_tree_attention_matches_definition(shape, L, kind, n):
    rng = np.random.default_rng(L * 31 + n)
    s = _session(shape)
    prompt = synth.motif_prompt(3000 + L, L + 1, 4, 16, 0.1, shape.vocab)
    s.prefill(_dev(prompt), max_new=8)
    tok, parent = _tree(kind, rng, n, shape.vocab)
    s.set_tree([int(t) for t in tok], [int(p) for p in parent])
    s.tree_verify_step(n)   # writes the nodes' K/V to slots L .. L+n-1
    Hq, Hkv, D = shape.n_heads, shape.n_kv_heads, shape.head_dim
    # queries with per-head sharpness: some heads spread, some peak on a few keys
    sharp = np.repeat(rng.uniform(0.5, 8.0, (1, Hq, 1)), n, axis=0)
    q = (rng.standard_normal((n, Hq, D)) * sharp / np.sqrt(D)).astype(np.float32)
    out = torch.empty((n, Hq * D), dtype=torch.float32, device="cuda")
    s.attention(0, n, torch.from_numpy(q).cuda(), out)
    kd = torch.empty((Hkv, L + n, D), dtype=torch.float32, device="cuda")
    vd = torch.empty_like(kd)
    s.copy_kv(0, 0, L + n, kd, vd)
    torch.cuda.synchronize()
    K, V = kd.cpu().numpy(), vd.cpu().numpy()
    ref = OS.tree_attention(q.astype(np.float64), K, V, L, parent).reshape(n, Hq * D)
    err = np.abs(out.cpu().numpy().astype(np.float64) - ref)
    bound = ATOL_V * np.abs(V).max()
    assert err.max() <= bound, (err.max(), bound, np.unravel_index(err.argmax(), err.shape))


def test_attention_entry_rejects_bad_arguments():
    shape = D64G7
    s = _session(shape)
    s.prefill(_dev(synth.motif_prompt(3001, 40, 4, 16, 0.1, shape.vocab)), max_new=8)
    s.set_tree([1, 2, 3], [-1, 0, 1])
    q = torch.zeros((16, shape.n_heads, shape.head_dim), device="cuda")
    out = torch.empty((16, shape.n_heads * shape.head_dim), device="cuda")
    with pytest.raises(W.W4A8Error):
        s.attention(0, 4, q, out)   # more nodes than the tree holds
    with pytest.raises(W.W4A8Error):
        s.attention(1, 3, q, out)   # no such layer
    s.attention(0, 3, q, out)       # zero queries: the mean of each node's visible values
    torch.cuda.synchronize()


def _forced_sequential_logits(shape, tokens):
    """Single-token steps over `tokens` (teacher-forced): logits after each token."""
    s = _session(shape)
    s.prefill(_dev(tokens[:1]), max_new=len(tokens) + 4)
    lg = torch.empty((1, shape.vocab), dtype=torch.float32, device="cuda")
    out = []
    for tok in tokens:
        s.set_tree([int(tok)], [-1])
        s.tree_verify_step(1, lg)
        out.append(lg[0].clone())
        s.accept_greedy(1)
    torch.cuda.synchronize()
    return torch.stack(out), s


@pytest.mark.parametrize("plen", [186, 193])
def test_verify_bitwise_equals_single_steps_d128(plen):
    # 16 tree nodes in one pass give the bits of single-token steps along every root path
    shape = D128
    prompt = list(synth.motif_prompt(3100 + plen, plen, 4, 16, 0.1, shape.vocab))
    rng = np.random.default_rng(plen)
    tok, parent = synth.random_tree(rng, 16, shape.vocab, max_depth=8)
    s = _session(shape)
    s.prefill(_dev(prompt), max_new=8)
    s.set_tree(tok.tolist(), parent.tolist())
    lg = torch.empty((16, shape.vocab), dtype=torch.float32, device="cuda")
    s.tree_verify_step(16, lg)
    torch.cuda.synchronize()
    leaves = [i for i in range(16) if i not in set(parent.tolist())]
    for leaf in leaves[:3]:
        path = OS.ancestors_or_self(parent, leaf)
        seq, _ = _forced_sequential_logits(shape, prompt[:-1] + [int(tok[j]) for j in path])
        for depth, node in enumerate(path):
            assert torch.equal(lg[node], seq[len(prompt) - 1 + depth]), (leaf, node)


def test_prefill_kv_bitwise_equals_sequential_kv_d128():
    # chains of 16 through the verification kernels write the bits of single steps
    shape = D128
    prompt = list(synth.motif_prompt(3200, 150, 4, 16, 0.1, shape.vocab))
    s = _session(shape)
    s.prefill(_dev(prompt), max_new=8)
    _, seq = _forced_sequential_logits(shape, prompt[:-1])
    n = len(prompt) - 1
    dims = (shape.n_kv_heads, n, shape.head_dim)
    k1, v1, k2, v2 = (torch.empty(dims, dtype=torch.float32, device="cuda") for _ in range(4))
    s.copy_kv(0, 0, n, k1, v1)
    seq.copy_kv(0, 0, n, k2, v2)
    torch.cuda.synchronize()
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
