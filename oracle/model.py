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
quantity is computed row by row, so a token's result does not depend on how
many tokens share the call.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import quant as Q

import synth


@dataclasses.dataclass
class Weights:
    shape: "synth.ModelShape"
    layers: list          # per layer: dict kind -> (codes int8 [rows][cols], scales fp16 [rows][cols/32])
    embed: tuple
    lm_head: tuple


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


def decision_margin(x: np.ndarray) -> float:
    """Distance, in code units, from the closest int8 decision of quant_row(x) to a rounding
    boundary (k + 1/2).  A second evaluation whose inputs differ in the last bits can only
    take a different code where this is small.  Diagnostic only."""
    x32 = np.asarray(x, dtype=np.float32)
    _, s = Q.quantize_act_per_token(x32[None, :])
    if s[0] == 0:
        return np.inf
    r = np.abs(x32.astype(np.float64)) / np.float64(s[0])
    r = r[r < 127.0]
    if r.size == 0:
        return np.inf
    return float(np.min(np.abs(r - np.floor(r) - 0.5)))


class Model:
    """A quantised decoder with an fp32 KV cache of ``kv_cap`` slots per layer."""

    def __init__(self, weights: Weights, kv_cap: int):
        self.w = weights
        self.shape = sh = weights.shape
        self.kv_cap = kv_cap
        self.K = [np.zeros((sh.n_kv_heads, kv_cap, sh.head_dim), np.float32) for _ in range(sh.n_layers)]
        self.V = [np.zeros((sh.n_kv_heads, kv_cap, sh.head_dim), np.float32) for _ in range(sh.n_layers)]
        self._dq = {}
        # diagnostic: smallest int8 decision margin of the token held in each cache slot
        self.margin = np.full(kv_cap, np.inf)
        self._m = np.inf

    # -- weights -----------------------------------------------------------
    def _deq(self, key, qs):
        if key not in self._dq:
            self._dq[key] = Q.dequantize_weights(qs[0], qs[1])
        return self._dq[key]

    def linear(self, key, qs, x_row: np.ndarray) -> np.ndarray:
        """W4A8 product of one activation row: quantise, then the exact-operand fp64 product."""
        self._m = min(self._m, decision_margin(x_row))
        q, s = quant_row(x_row)
        a = q.astype(np.float64) * np.float64(s)
        return self._deq(key, qs) @ a

    def embed(self, tok: int) -> np.ndarray:
        q, s = self.w.embed
        H = self.shape.hidden
        return q[tok].astype(np.float64) * np.repeat(s[tok].astype(np.float64), Q.GROUP)[:H]

    # -- forward -------------------------------------------------------------
    def forward(self, toks, pos, slots, visible, trace=None) -> np.ndarray:
        """Evaluate tokens ``toks`` at logical positions ``pos``; write their K/V to cache
        ``slots``; token i attends to the cache slots ``visible[i]`` (given in logical
        order, all written before attention).  Returns fp64 logits [n][vocab].
        ``trace`` (a dict) collects per-layer intermediates for the tests."""
        sh = self.shape
        n = len(toks)
        H, Hq, Hkv, d = sh.hidden, sh.n_heads, sh.n_kv_heads, sh.head_dim
        x = np.stack([self.embed(int(t)) for t in toks])
        tok_m = np.full(n, np.inf)
        for l, Wl in enumerate(self.w.layers):
            qh = np.zeros((n, Hq, d))
            for i in range(n):
                self._m = tok_m[i]
                n1 = rmsnorm(x[i], sh.rms_eps)
                qv = self.linear((l, synth.T_WQ), Wl[synth.T_WQ], n1).reshape(Hq, d)
                kv = self.linear((l, synth.T_WK), Wl[synth.T_WK], n1).reshape(Hkv, d)
                vv = self.linear((l, synth.T_WV), Wl[synth.T_WV], n1).reshape(Hkv, d)
                qh[i] = rope(qv, int(pos[i]), sh.rope_base)
                self.K[l][:, int(slots[i])] = rope(kv, int(pos[i]), sh.rope_base).astype(np.float32)
                self.V[l][:, int(slots[i])] = vv.astype(np.float32)
                tok_m[i] = self._m
            for i in range(n):
                self._m = tok_m[i]
                vis = np.asarray(visible[i], dtype=np.int64)
                att = np.zeros((Hq, d))
                for h in range(Hq):
                    kh = kv_head_of(h, Hq, Hkv)
                    att[h] = attend(qh[i, h], self.K[l][kh, vis], self.V[l][kh, vis])
                hrow = x[i] + self.linear((l, synth.T_WO), Wl[synth.T_WO], att.reshape(-1))
                mlp = self.mlp(l, Wl, rmsnorm(hrow, sh.rms_eps))
                if trace is not None:
                    trace.setdefault("att", []).append(att.copy())
                    trace.setdefault("h", []).append(hrow.copy())
                    trace.setdefault("mlp", []).append(mlp.copy())
                x[i] = hrow + mlp
                tok_m[i] = self._m
        logits = np.zeros((n, sh.vocab))
        for i in range(n):
            self._m = tok_m[i]
            logits[i] = self.linear("lm", self.w.lm_head, rmsnorm(x[i], sh.rms_eps))
            tok_m[i] = self._m
            self.margin[int(slots[i])] = tok_m[i]
        return logits

    def mlp(self, l, Wl, n2) -> np.ndarray:
        """SwiGLU block on a normalised row: quant(silu(gate) * up) -> down projection."""
        g = self.linear((l, synth.T_WG), Wl[synth.T_WG], n2)
        u = self.linear((l, synth.T_WU), Wl[synth.T_WU], n2)
        return self.linear((l, synth.T_WD), Wl[synth.T_WD], silu(g) * u)

    # -- protocols -------------------------------------------------------------
    def prefill(self, toks) -> np.ndarray:
        """Causal pass over ``toks`` at positions/slots 0..n-1."""
        n = len(toks)
        return self.forward(toks, list(range(n)), list(range(n)), [list(range(i + 1)) for i in range(n)])

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
        m.prefill(prompt[:-1])
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
