"""Seeded input generators (no method arithmetic here).

Counter-based stream
--------------------
Every large tensor is drawn from a counter-based generator so that any slice of
it can be reproduced independently, on the host (numpy, this file) or on the
device (``synth.cu``).  The generator is the SplitMix64 output function of
Steele, Lea and Flood, "Fast Splittable Pseudorandom Number Generators"
(OOPSLA 2014), applied to a Weyl sequence:

    fin(z)   = z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
               z ^= z >> 27; z *= 0x94D049BB133111EB; z ^ (z >> 31)
    sm64(k, i) = fin(k + (i + 1) * 0x9E3779B97F4A7C15)        (mod 2**64)
    key(seed, stream) = sm64(sm64(seed, 0), stream)

Draws built on it (all integer until one final IEEE fp32 operation, so that
numpy and CUDA agree bit for bit):

* ``normal``: element e takes words sm64(key, 3e), sm64(key, 3e+1),
  sm64(key, 3e+2), splits them into twelve 16-bit integers u_j and returns
  fp32(S - 393210) * fp32(sigma / 65536) with S = sum_j u_j.  S - 393210 is the
  Irwin-Hall sum of 12 uniforms centred at zero with variance ~65536**2, so the
  value is approximately N(0, sigma**2) (bounded at +-6 sigma).
* ``uniform_codes``: element e takes nibble (e % 16) of word sm64(key, e // 16)
  and subtracts 8: uniform on {-8..7}.
* ``uniform_scales``: element e takes u = (sm64(key, e) >> 40) * 2**-24 in
  [0, 1), then fp16(fp32(fp32(u * (hi - lo)) + lo)) with both fp32 operations
  rounded separately (no fused multiply-add).
"""
from __future__ import annotations

import dataclasses
import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB


def _fin(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(M1)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(M2)
    return z ^ (z >> np.uint64(31))


def sm64(k: int, idx: np.ndarray) -> np.ndarray:
    """Word ``idx`` of the SplitMix64 stream with key ``k`` (uint64 array)."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(k & MASK64) + (idx + np.uint64(1)) * np.uint64(GOLDEN)
        return _fin(z)


def sm64_scalar(k: int, i: int) -> int:
    z = (k + (i + 1) * GOLDEN) & MASK64
    z ^= z >> 30
    z = (z * M1) & MASK64
    z ^= z >> 27
    z = (z * M2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    return sm64_scalar(sm64_scalar(seed & MASK64, 0), stream & MASK64)


def sigma_mult(sigma: float) -> np.float32:
    return np.float32(sigma / 65536.0)


def normal(seed: int, stream: int, start: int, count: int, sigma: float) -> np.ndarray:
    """Approximately N(0, sigma^2) fp32 values, elements [start, start+count)."""
    k = stream_key(seed, stream)
    out = np.empty(count, dtype=np.float32)
    mult = sigma_mult(sigma)
    step = 1 << 22
    for c0 in range(0, count, step):
        n = min(step, count - c0)
        e = np.arange(start + c0, start + c0 + n, dtype=np.uint64)
        s = np.zeros(n, dtype=np.int64)
        with np.errstate(over="ignore"):
            for j in range(3):
                w = sm64(k, np.uint64(3) * e + np.uint64(j))
                for b in range(4):
                    s += ((w >> np.uint64(16 * b)) & np.uint64(0xFFFF)).astype(np.int64)
        out[c0:c0 + n] = (s - 393210).astype(np.float32) * mult
    return out


def uniform_codes(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Uniform int4 codes in {-8..7} as int8: element e is nibble e % 16 of word e // 16."""
    k = stream_key(seed, stream)
    w0, w1 = start // 16, (start + count + 15) // 16
    out = np.empty((w1 - w0) * 16, dtype=np.int8)
    shifts = (np.uint64(4) * np.arange(16, dtype=np.uint64))[None, :]
    step = 1 << 20
    for c0 in range(w0, w1, step):
        c1 = min(w1, c0 + step)
        w = sm64(k, np.arange(c0, c1, dtype=np.uint64))
        nib = ((w[:, None] >> shifts) & np.uint64(15)).astype(np.int8) - np.int8(8)
        out[(c0 - w0) * 16:(c1 - w0) * 16] = nib.reshape(-1)
    off = start - w0 * 16
    return out[off:off + count].copy()


def uniform_scales(seed: int, stream: int, start: int, count: int,
                   lo: float = 0.001, hi: float = 0.02) -> np.ndarray:
    """fp16 values approximately uniform on [lo, hi)."""
    k = stream_key(seed, stream)
    e = np.arange(start, start + count, dtype=np.uint64)
    w = sm64(k, e)
    u = (w >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)
    v = (u * np.float32(hi - lo)).astype(np.float32)
    v = (v + np.float32(lo)).astype(np.float32)
    return v.astype(np.float16)


# --------------------------------------------------------------------------
# model shapes (the pages' workloads, synthetic random init)
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class ModelShape:
    name: str
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int            # FFN width as used by kernels (multiple of 32)
    ffn_real: int       # FFN width before zero padding
    vocab: int
    tied: bool
    rope_base: float = 10000.0
    rms_eps: float = 1e-6
    weight_sigma: float = 0.02

    @property
    def qkv_rows(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim


TINY = ModelShape("tiny-2L-256h", 2, 256, 4, 2, 64, 704, 688, 4096, False)
QWEN05B = ModelShape("qwen2.5-0.5b-shaped", 24, 896, 14, 2, 64, 4864, 4864, 151936, True)
LLAMA8B = ModelShape("llama3-8b-shaped", 32, 4096, 32, 8, 128, 14336, 14336, 128256, False)

SHAPES = {s.name: s for s in (TINY, QWEN05B, LLAMA8B)}

# tensor stream ids of the counter-based generator
T_WQ, T_WK, T_WV, T_WO, T_WG, T_WU, T_WD = range(7)
STREAM_EMBED = 1 << 20
STREAM_LM_HEAD = (1 << 20) + 1


def layer_stream(layer: int, kind: int) -> int:
    return layer * 16 + kind


def tensor_shape(shape: ModelShape, kind: int):
    """(rows, cols, real_rows, real_cols) of one layer tensor, [out][in]."""
    H, F, Fr = shape.hidden, shape.ffn, shape.ffn_real
    qd = shape.n_heads * shape.head_dim
    kvd = shape.n_kv_heads * shape.head_dim
    return {
        T_WQ: (qd, H, qd, H), T_WK: (kvd, H, kvd, H), T_WV: (kvd, H, kvd, H),
        T_WO: (H, qd, H, qd), T_WG: (F, H, Fr, H), T_WU: (F, H, Fr, H),
        T_WD: (H, F, H, Fr),
    }[kind]


def dense_weight(shape: ModelShape, seed: int, stream: int, rows: int, cols: int,
                 real_rows: int, real_cols: int, row0: int = 0, nrows: int | None = None) -> np.ndarray:
    """fp32 weight rows [row0, row0+nrows) of a [rows][cols] tensor.

    Element (r, c) with r < real_rows and c < real_cols is element r*real_cols+c of
    the ``normal`` stream; the zero padding beyond the real extent is exactly 0.
    """
    if nrows is None:
        nrows = rows - row0
    out = np.zeros((nrows, cols), dtype=np.float32)
    r_hi = min(row0 + nrows, real_rows)
    if r_hi > row0:
        vals = normal(seed, stream, row0 * real_cols, (r_hi - row0) * real_cols, shape.weight_sigma)
        out[: r_hi - row0, :real_cols] = vals.reshape(r_hi - row0, real_cols)
    return out


# --------------------------------------------------------------------------
# prompts and trees
# --------------------------------------------------------------------------

def motif_prompt(seed: int, length: int, n_motifs: int, motif_len: int, p_sub: float,
                 vocab: int) -> np.ndarray:
    """Motif-repeated prompt: motifs of i.i.d. uniform tokens, instances drawn
    uniformly with replacement and concatenated, truncated to ``length``; then each
    token is replaced with probability ``p_sub`` by a uniform token."""
    rng = np.random.default_rng(seed)
    motifs = rng.integers(0, vocab, size=(n_motifs, motif_len))
    n_inst = -(-length // motif_len)
    picks = rng.integers(0, n_motifs, size=n_inst)
    toks = motifs[picks].reshape(-1)[:length].copy()
    sub = rng.random(length) < p_sub
    toks[sub] = rng.integers(0, vocab, size=int(sub.sum()))
    return toks.astype(np.int32)


def random_tree(rng: np.random.Generator, n: int, vocab: int, n_valid: int | None = None,
                max_depth: int | None = None):
    """Random tree: parent[i] < i, parent[0] = -1.  Returns (tok, parent)."""
    if n_valid is None:
        n_valid = n
    tok = rng.integers(0, vocab, size=n).astype(np.int32)
    parent = np.zeros(n, dtype=np.int32)
    parent[0] = -1
    depth = np.zeros(n, dtype=np.int32)
    for i in range(1, n):
        if i < n_valid:
            while True:
                p = int(rng.integers(0, i))
                if max_depth is None or depth[p] + 1 <= max_depth:
                    break
        else:
            p = 0
        parent[i] = p
        depth[i] = depth[p] + 1
    return tok, parent


def matmul_case(seed: int, M: int, K: int, N: int):
    """Matmul sweep inputs: int4 codes U{-8..7} [N][K], fp16 scales U(0.001,0.02)
    [N][K/32], activations ~N(0,1) fp32 [M][K].  Streams 1, 2, 3 of ``seed``."""
    q = uniform_codes(seed, 1, 0, N * K).reshape(N, K)
    s = uniform_scales(seed, 2, 0, N * (K // 32)).reshape(N, K // 32)
    x = normal(seed, 3, 0, M * K, 1.0).reshape(M, K)
    return q, s, x


def matmul_rows(seed: int, K: int, rows: np.ndarray):
    """Codes and scales of selected rows of the ``matmul_case`` weight matrix."""
    qs, ss = [], []
    for r in np.asarray(rows).tolist():
        qs.append(uniform_codes(seed, 1, r * K, K))
        ss.append(uniform_scales(seed, 2, r * (K // 32), K // 32))
    return np.stack(qs), np.stack(ss)
