"""The quantised decoder evaluated by definition, and greedy decoding with it.

"GPU-Resident Speculative Decoding ...":
* Design > Small-Batch Verification Kernels: every matrix multiplication takes
  int4 g32 weights and int8 activations quantised right before it; the
  activation quantisation follows the RMSNorm and SiLU steps.
* Implementation: the KV cache is kept in 32-bit floats; speculation must
  reproduce the greedy decoding of the same quantised runtime.
* Design > GPU-Resident Speculation Loop: in a verification step each tree node
  attends to the committed cache and to its ancestors.

Layer (Llama/Qwen style, no biases, RMSNorm gain 1):
    n1 = quant(rmsnorm(x));  q, k, v = n1 Wq, n1 Wk, n1 Wv;  rope(q), rope(k)
    h  = x + quant(attn(q, K, V)) Wo
    n2 = quant(rmsnorm(h));  x' = h + quant(silu(n2 Wg) * (n2 Wu)) Wd
    logits = quant(rmsnorm(x_L)) W_lm        (W_lm = embedding table when tied)
rmsnorm(x) = x / sqrt(mean(x^2) + eps); silu(z) = z / (1 + exp(-z));
attention = softmax(q.k / sqrt(d)) v over the visible keys, query head h reading
KV head h // (Hq / Hkv); rope is rotate-half with theta_i = base^(-2i/d).

Arithmetic is fp64; K and V are stored in fp32 (the pages' KV precision); the
int8 code decisions are taken in fp32 (``oracle.quant``).  Every per-token
quantity is computed row by row (each row quantised on its own, each product a
matrix-vector product), so a token's result does not depend on how many tokens
share the call.

Quantisation points ("stages") of one token, in evaluation order: for every layer
l, ``l{l}.n1`` (RMSNorm output before Q/K/V), ``l{l}.att`` (attention output before
O), ``l{l}.n2`` (RMSNorm output before gate/up), ``l{l}.sw`` (SwiGLU output before
down); then ``lm`` (final RMSNorm output before the LM head).  With ``record`` set,
the model keeps, per (cache slot, stage), the int8 codes and the distance of every
code's decision to its rounding boundary (``decision_margins``).
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import quant as Q

import synth

# dequantised weights are cached while the model's total stays below this; larger
# models dequantise each product in row blocks (same values, bounded memory)
DEQ_CACHE_BYTES = 1 << 30
DEQ_BLOCK_ELEMS = 1 << 25


@dataclasses.dataclass
class Weights:
    shape: "synth.ModelShape"
    layers: list          # per layer: dict kind -> (codes int8 [rows][cols], scales fp16 [rows][cols/32])
    embed: tuple
    lm_head: tuple
    # dequantised fp64 weights shared by the Models built on these weights (when cached)
    deq_cache: dict = dataclasses.field(default_factory=dict, repr=False)


def build_weights(shape, seed: int) -> Weights:
    """Seeded random-init weights (synth's counter-based normal stream, sigma=0.02),
    quantised by the oracle's own weight quantiser."""
    layers = []
    for layer in range(shape.n_layers):
        d = {}
        for kind in (synth.T_WQ, synth.T_WK, synth.T_WV, synth.T_WO, synth.T_WG, synth.T_WU, synth.T_WD):
            rows, cols, rr, rc = synth.tensor_shape(shape, kind)
            w = synth.dense_weight(shape, seed, synth.layer_stream(layer, kind), rows, cols, rr, rc)
            d[kind] = Q.quantize_weights_g32(w)
        layers.append(d)
    V, H = shape.vocab, shape.hidden
    emb = Q.quantize_weights_g32(synth.dense_weight(shape, seed, synth.STREAM_EMBED, V, H, V, H))
    if shape.tied:
        lm = emb
    else:
        lm = Q.quantize_weights_g32(synth.dense_weight(shape, seed, synth.STREAM_LM_HEAD, V, H, V, H))
    return Weights(shape, layers, emb, lm)


def stage_names(n_layers: int) -> list:
    """The quantisation points of one token in evaluation order."""
    out = []
    for l in range(n_layers):
        out += ["l%d.n1" % l, "l%d.att" % l, "l%d.n2" % l, "l%d.sw" % l]
    return out + ["lm"]


def stage_width(shape, stage: str) -> int:
    """Inputs quantised at a stage."""
    if stage.endswith(".att"):
        return shape.n_heads * shape.head_dim
    if stage.endswith(".sw"):
        return shape.ffn
    return shape.hidden


def rmsnorm(x: np.ndarray, eps: float) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x) + eps)


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def rope(v: np.ndarray, pos: int, base: float) -> np.ndarray:
    """Rotate-half RoPE of one head vector (fp64) at position ``pos``."""
    d = v.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    theta = base ** (-2.0 * i / d)
    ang = pos * theta
    c, s = np.cos(ang), np.sin(ang)
    v1, v2 = v[..., :half], v[..., half:]
    return np.concatenate([v1 * c - v2 * s, v2 * c + v1 * s], axis=-1)


def attend(q: np.ndarray, Kv: np.ndarray, Vv: np.ndarray) -> np.ndarray:
    """softmax(K q / sqrt(d)) V for one query head over the visible keys (fp64)."""
    d = q.shape[-1]
    sc = (np.asarray(Kv, dtype=np.float64) @ q) / np.sqrt(d)
    p = np.exp(sc - sc.max())
    return (p @ np.asarray(Vv, dtype=np.float64)) / p.sum()


def kv_head_of(h: int, n_heads: int, n_kv_heads: int) -> int:
    """Grouped-query attention: consecutive groups of Hq/Hkv query heads share a KV head."""
    return h // (n_heads // n_kv_heads)


def quant_row(x: np.ndarray):
    """Per-token int8 quantisation of one fp64 row; the decision is taken in fp32."""
    q, s = Q.quantize_act_per_token(np.asarray(x, dtype=np.float32)[None, :])
    return q[0], s[0]


def decision_margins(x: np.ndarray) -> np.ndarray:
    """Per input of quant_row(x): the distance, in code units, of its fp32 quotient
    r = |x_k| / s from the nearest rounding boundary k + 1/2 of the round-to-nearest
    decision (0.5 = the middle between two boundaries).  Inputs whose quotient reaches
    the clamp at 127 have no rounding boundary above it and take the distance to the one
    below.  A second evaluation of the same definition whose inputs differ from these by
    less than the margin (in code units) takes the same code.  An all-zero row has no
    decision (infinite margins)."""
    x32 = np.asarray(x, dtype=np.float32)
    _, s = Q.quantize_act_per_token(x32[None, :])
    if s[0] == 0:
        return np.full(x32.shape, np.inf)
    r = np.abs(x32.astype(np.float64)) / np.float64(s[0])
    r = np.minimum(r, 127.0)
    return np.abs(r - np.floor(r) - 0.5)


def decision_margin(x: np.ndarray) -> float:
    """Smallest of ``decision_margins(x)``."""
    return float(np.min(decision_margins(x)))


class Model:
    """A quantised decoder with an fp32 KV cache of ``kv_cap`` slots per layer."""

    def __init__(self, weights: Weights, kv_cap: int, record: bool = False, cache_bytes=None):
        self.w = weights
        self.shape = sh = weights.shape
        self.kv_cap = kv_cap
        self.K = [np.zeros((sh.n_kv_heads, kv_cap, sh.head_dim), np.float32) for _ in range(sh.n_layers)]
        self.V = [np.zeros((sh.n_kv_heads, kv_cap, sh.head_dim), np.float32) for _ in range(sh.n_layers)]
        self._dq = weights.deq_cache
        total = sum(q.size for d in weights.layers for q, _ in d.values()) + weights.lm_head[0].size
        self._cache_deq = total * 8 <= (DEQ_CACHE_BYTES if cache_bytes is None else cache_bytes)
        # (slot, stage) -> (codes int8 [K], margins fp64 [K]) of the last evaluation at that slot
        self.record = {} if record else None

    # -- weights -----------------------------------------------------------
    def _deq(self, key, qs, r0=None, r1=None):
        if r0 is None:
            if self._cache_deq:
                if key not in self._dq:
                    self._dq[key] = Q.dequantize_weights(qs[0], qs[1])
                return self._dq[key]
            return Q.dequantize_weights(qs[0], qs[1])
        if self._cache_deq:
            return self._deq(key, qs)[r0:r1]
        return Q.dequantize_weights(qs[0][r0:r1], qs[1][r0:r1])

    def products(self, key, qs, A: np.ndarray) -> np.ndarray:
        """W4A8 products of already quantised (dequantised, exact in fp64) activation rows
        A [n][K]: every row is its own matrix-vector product with the fp64 weights."""
        rows, cols = qs[0].shape
        n = A.shape[0]
        out = np.zeros((n, rows))
        blk = max(1, DEQ_BLOCK_ELEMS // cols)
        for r0 in range(0, rows, blk):
            r1 = min(rows, r0 + blk)
            Wb = self._deq(key, qs, r0, r1)
            for i in range(n):
                out[i, r0:r1] = Wb @ A[i]
        return out

    def quantize(self, X: np.ndarray, stage=None, slots=None) -> np.ndarray:
        """Per-row int8 quantisation (decisions in fp32); returns the dequantised rows
        (codes times scale, exact in fp64).  Records codes and margins when enabled."""
        out = np.zeros(X.shape)
        for i in range(X.shape[0]):
            q, s = quant_row(X[i])
            out[i] = q.astype(np.float64) * np.float64(s)
            if self.record is not None and stage is not None:
                self.record[(int(slots[i]), stage)] = (q.copy(), decision_margins(X[i]))
        return out

    def linear(self, key, qs, x_row: np.ndarray) -> np.ndarray:
        """W4A8 product of one activation row: quantise, then the exact-operand fp64 product."""
        return self.products(key, qs, self.quantize(np.asarray(x_row, dtype=np.float64)[None, :]))[0]

    def embed(self, tok: int) -> np.ndarray:
        q, s = self.w.embed
        H = self.shape.hidden
        return q[tok].astype(np.float64) * np.repeat(s[tok].astype(np.float64), Q.GROUP)[:H]

    # -- forward -------------------------------------------------------------
    def forward(self, toks, pos, slots, visible, trace=None, head: bool = True):
        """Evaluate tokens ``toks`` at logical positions ``pos``; write their K/V to cache
        ``slots``; token i attends to the cache slots ``visible[i]`` (given in logical
        order, all written before attention).  Returns fp64 logits [n][vocab] (None when
        ``head`` is False).  ``trace`` (a dict) collects per-layer intermediates for the
        tests."""
        sh = self.shape
        n = len(toks)
        H, Hq, Hkv, d = sh.hidden, sh.n_heads, sh.n_kv_heads, sh.head_dim
        eps = sh.rms_eps
        x = np.stack([self.embed(int(t)) for t in toks])
        for l, Wl in enumerate(self.w.layers):
            A = self.quantize(np.stack([rmsnorm(x[i], eps) for i in range(n)]), "l%d.n1" % l, slots)
            qv = self.products((l, synth.T_WQ), Wl[synth.T_WQ], A).reshape(n, Hq, d)
            kv = self.products((l, synth.T_WK), Wl[synth.T_WK], A).reshape(n, Hkv, d)
            vv = self.products((l, synth.T_WV), Wl[synth.T_WV], A).reshape(n, Hkv, d)
            qh = np.zeros((n, Hq, d))
            for i in range(n):
                qh[i] = rope(qv[i], int(pos[i]), sh.rope_base)
                self.K[l][:, int(slots[i])] = rope(kv[i], int(pos[i]), sh.rope_base).astype(np.float32)
                self.V[l][:, int(slots[i])] = vv[i].astype(np.float32)
            att = np.zeros((n, Hq, d))
            for i in range(n):
                vis = np.asarray(visible[i], dtype=np.int64)
                for h in range(Hq):
                    kh = kv_head_of(h, Hq, Hkv)
                    att[i, h] = attend(qh[i, h], self.K[l][kh, vis], self.V[l][kh, vis])
            A = self.quantize(att.reshape(n, Hq * d), "l%d.att" % l, slots)
            hrow = x + self.products((l, synth.T_WO), Wl[synth.T_WO], A)
            A = self.quantize(np.stack([rmsnorm(hrow[i], eps) for i in range(n)]), "l%d.n2" % l, slots)
            g = self.products((l, synth.T_WG), Wl[synth.T_WG], A)
            u = self.products((l, synth.T_WU), Wl[synth.T_WU], A)
            A = self.quantize(silu(g) * u, "l%d.sw" % l, slots)
            mlp = self.products((l, synth.T_WD), Wl[synth.T_WD], A)
            if trace is not None:
                for i in range(n):
                    trace.setdefault("att", []).append(att[i].copy())
                    trace.setdefault("h", []).append(hrow[i].copy())
                    trace.setdefault("mlp", []).append(mlp[i].copy())
            x = hrow + mlp
        if not head:
            return None
        A = self.quantize(np.stack([rmsnorm(x[i], eps) for i in range(n)]), "lm", slots)
        return self.products("lm", self.w.lm_head, A)

    def mlp(self, l, Wl, n2) -> np.ndarray:
        """SwiGLU block on a normalised row: quant(silu(gate) * up) -> down projection."""
        g = self.linear((l, synth.T_WG), Wl[synth.T_WG], n2)
        u = self.linear((l, synth.T_WU), Wl[synth.T_WU], n2)
        return self.linear((l, synth.T_WD), Wl[synth.T_WD], silu(g) * u)

    # -- protocols -------------------------------------------------------------
    def prefill(self, toks, head: bool = True):
        """Causal pass over ``toks`` at positions/slots 0..n-1."""
        n = len(toks)
        return self.forward(toks, list(range(n)), list(range(n)), [list(range(i + 1)) for i in range(n)],
                            head=head)

    def step(self, tok: int, L: int) -> np.ndarray:
        """One plain decoding step: token at position/slot L attending to slots 0..L."""
        return self.forward([tok], [L], [L], [list(range(L + 1))])[0]


def argmax_lowest(v: np.ndarray) -> int:
    """argmax with ties going to the lowest index."""
    return int(np.argmax(v))


def greedy_decode(weights: Weights, prompt, max_new: int, eos: int = -1, kv_cap: int | None = None):
    """Plain greedy decoding: prefill prompt[:-1], then one token per step starting from
    the last prompt token.  Returns (tokens, per-step fp64 logits)."""
    prompt = [int(t) for t in prompt]
    n = len(prompt)
    m = Model(weights, kv_cap or (n + max_new + 1))
    if n > 1:
        m.prefill(prompt[:-1], head=False)
    L, tok = n - 1, prompt[-1]
    out, logits = [], []
    while len(out) < max_new:
        lg = m.step(tok, L)
        logits.append(lg)
        tok = argmax_lowest(lg)
        out.append(tok)
        L += 1
        if tok == eos:
            break
    return out, logits


def teacher_forced_logits(weights: Weights, prompt, forced, kv_cap: int | None = None):
    """Logits of plain decoding steps whose inputs are the given tokens: prefill
    prompt[:-1], then steps on prompt[-1], forced[0], forced[1], ...  Returns the
    fp64 logits of each step (len(forced) + 1 rows)."""
    prompt = [int(t) for t in prompt]
    n = len(prompt)
    m = Model(weights, kv_cap or (n + len(forced) + 2))
    if n > 1:
        m.prefill(prompt[:-1], head=False)
    out = []
    L = n - 1
    for tok in [prompt[-1]] + [int(t) for t in forced]:
        out.append(m.step(tok, L))
        L += 1
    return out
