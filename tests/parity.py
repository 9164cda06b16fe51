"""Helpers of the GPU parity tests: the code-level comparison of a verification pass.

The benchmark spec's bound on logits is max |gpu - oracle| <= 2e-3 * (max - min of the oracle
row).  Every matrix product consumes int8 activation codes that are quantised right before
it ("GPU-Resident Speculative Decoding ...", Design > Small-Batch Verification Kernels), and
a code is a discontinuous function of the fp32 value it rounds: where the oracle's value
lies within the kernels' rounding error of a boundary k + 1/2, the GPU may take the
neighbouring code, and that one-step difference then moves everything downstream of it by
far more than rounding does.  So the comparison is made at the level of the codes:

* ``w4a8_tree_verify_trace`` returns every code the GPU's matmuls consumed; the oracle
  records its own codes and, per code, the distance of its decision to the boundary.
* A *first flip* is a code that differs while every code it depends on (earlier stages of
  the node and of its ancestors) agrees.  Each first flip must differ by one step and sit
  within ``DELTA_FLIP`` code units of a boundary: the GPU may only resolve a decision the
  fp32 arithmetic cannot decide differently from the oracle.
* A row whose dependency cone holds no differing code must meet the benchmark spec's bound
  ``REL_TOL``; a row downstream of a flip must meet ``REL_TOL_FLIP``; a greedy token must
  agree wherever the oracle's top-2 margin exceeds twice the row's bound.
* The context (cache slots below the committed length) is either given to both sides as the
  same fp32 K/V (``w4a8_session_load_kv``), or computed by each side, in which case it counts
  as clean only where the GPU's cached K/V equal the oracle's to ``KV_REL`` (a flipped code in
  the context moves the K/V of its token by about one code step, 1/127 of the row's range).
"""
from __future__ import annotations

import numpy as np

import synth
from oracle import model as OM
from oracle import spec as OS

REL_TOL = 2e-3
REL_TOL_FLIP = 2e-2
DELTA_FLIP = 2e-3
KV_REL = 1e-4


def stage_blocks(shape, N):
    """(stage, inputs, byte offset) of the trace of a pass over N tokens."""
    out, off = [], 0
    for st in OM.stage_names(shape.n_layers):
        K = OM.stage_width(shape, st)
        out.append((st, K, off))
        off += N * K
    return out, off


def split_trace(codes: np.ndarray, shape, N) -> dict:
    blocks, total = stage_blocks(shape, N)
    assert codes.size >= total
    return {st: codes[off:off + N * K].reshape(N, K) for st, K, off in blocks}


class Flips:
    """Code comparison of one verification pass of N nodes at slots L..L+N-1."""

    def __init__(self, gpu_codes: dict, record: dict, shape, L: int, parent):
        self.stages = OM.stage_names(shape.n_layers)
        N = len(parent)
        self.N = N
        self.paths = [OS.ancestors_or_self(parent, i) for i in range(N)]
        self.mism = {}   # (node, stage index) -> (index array, gpu codes, oracle codes, margins)
        for i in range(N):
            for j, st in enumerate(self.stages):
                oq, om = record[(L + i, st)]
                g = gpu_codes[st][i]
                d = np.flatnonzero(g.astype(np.int32) != oq.astype(np.int32))
                if d.size:
                    self.mism[(i, j)] = (d, g[d].astype(np.int32), oq[d].astype(np.int32), om[d])

    def _dirty_before(self, i, j):
        return any((a, jj) in self.mism for a in self.paths[i] for jj in range(j))

    def first_flips(self):
        """Mismatches whose inputs all agree: list of (node, stage, idx, gpu, oracle, margin)."""
        out = []
        for (i, j), (d, g, o, m) in sorted(self.mism.items()):
            if not self._dirty_before(i, j):
                for k in range(d.size):
                    out.append((i, self.stages[j], int(d[k]), int(g[k]), int(o[k]), float(m[k])))
        return out

    def row_clean(self, i):
        """No differing code in the cone of node i's logits (its own stages, its ancestors'
        stages before the LM head)."""
        last = len(self.stages) - 1
        for a in self.paths[i]:
            top = last + 1 if a == i else last
            if any((a, j) in self.mism for j in range(top)):
                return False
        return True

    def check_first_flips(self):
        ff = self.first_flips()
        for (i, st, k, g, o, m) in ff:
            assert abs(g - o) == 1, ("first flip of more than one step", i, st, k, g, o, m)
            assert m < DELTA_FLIP, ("first flip away from a rounding boundary", i, st, k, g, o, m)
        return ff


def kv_clean(gpu_k, gpu_v, ref_k, ref_v) -> np.ndarray:
    """Per cache slot: the GPU's K and V equal the oracle's within KV_REL of each head row's
    largest magnitude.  Arrays [Hkv][slots][d]."""
    ok = np.ones(gpu_k.shape[1], dtype=bool)
    for g, r in ((gpu_k, ref_k), (gpu_v, ref_v)):
        g = g.astype(np.float64)
        r = r.astype(np.float64)
        scale = np.abs(r).max(axis=2, keepdims=True) + 1e-30
        ok &= (np.abs(g - r) <= KV_REL * scale).all(axis=(0, 2))
    return ok


def check_rows(gpu, ref, pred, clean):
    """Row bounds and greedy-token agreement; returns (rows at REL_TOL, rows at REL_TOL_FLIP)."""
    strict = loose = 0
    for i in range(ref.shape[0]):
        rng = ref[i].max() - ref[i].min()
        rel = REL_TOL if clean[i] else REL_TOL_FLIP
        bound = rel * rng
        err = np.abs(gpu[i].astype(np.float64) - ref[i]).max()
        assert err <= bound, (i, bool(clean[i]), err / rng)
        if pred is not None:
            top2 = np.sort(ref[i])[-2:]
            if top2[1] - top2[0] > 2 * bound:
                assert pred[i] == int(np.argmax(ref[i])), i
        if clean[i]:
            strict += 1
        else:
            loose += 1
    return strict, loose


class Tally:
    """Rows checked at each bound over a test module; reported and asserted at its end."""

    def __init__(self):
        self.strict = 0
        self.loose = 0
        self.first_flips = []

    def add(self, strict, loose, ff=()):
        self.strict += strict
        self.loose += loose
        self.first_flips += list(ff)

    def summary(self):
        m = max((f[5] for f in self.first_flips), default=None)
        return ("rows at the 2e-3 bound: %d, downstream of a code flip (2e-2): %d; first flips: %d, "
                "largest margin %s" % (self.strict, self.loose, len(self.first_flips), m))


# ------------------------------------------------------------ GPU-side helpers (need torch)

def traced_verify(s, shape, N):
    """tree_verify_trace of N nodes: (logits [N][V] fp32, codes per stage, pred)."""
    codes = _torch().empty(s.trace_bytes(N), dtype=_torch().int8, device="cuda")
    lg = _torch().empty((N, shape.vocab), dtype=_torch().float32, device="cuda")
    s.tree_verify_trace(N, codes, lg)
    pred = s.pred(N)
    return lg.cpu().numpy(), split_trace(codes.cpu().numpy(), shape, N), pred


def gpu_kv(s, shape, n):
    ks, vs = [], []
    for layer in range(shape.n_layers):
        k = _torch().empty((shape.n_kv_heads, n, shape.head_dim), dtype=_torch().float32, device="cuda")
        v = _torch().empty_like(k)
        s.copy_kv(layer, 0, n, k, v)
        ks.append(k)
        vs.append(v)
    _torch().cuda.synchronize()
    return [k.cpu().numpy() for k in ks], [v.cpu().numpy() for v in vs]


def ctx_clean(s, shape, om, L):
    """All cached slots below L hold the oracle's K/V (to KV_REL) in every layer."""
    if L == 0:
        return True
    ks, vs = gpu_kv(s, shape, L)
    return all(kv_clean(ks[l], vs[l], om.K[l][:, :L], om.V[l][:, :L]).all() for l in range(shape.n_layers))


def synthetic_kv(shape, seed, L):
    """Seeded fp32 K and V [layers][Hkv][L][d], N(0, 1): the same cache for both sides."""
    n = shape.n_kv_heads * L * shape.head_dim
    ks = [synth.normal(seed, 2 * l, 0, n, 1.0).reshape(shape.n_kv_heads, L, shape.head_dim)
          for l in range(shape.n_layers)]
    vs = [synth.normal(seed, 2 * l + 1, 0, n, 1.0).reshape(shape.n_kv_heads, L, shape.head_dim)
          for l in range(shape.n_layers)]
    return ks, vs


def verify_on_given_cache(s, ow, shape, L, tok, parent, kv_seed, tally):
    """Tree verification over a given cache of L slots (the same fp32 K/V loaded into the
    session and the oracle): code-level parity of the N rows."""
    N = len(tok)
    ks, vs = synthetic_kv(shape, kv_seed, L)
    if L > 0:
        for l in range(shape.n_layers):
            s.load_kv(l, 0, L, _torch().from_numpy(ks[l]).cuda(), _torch().from_numpy(vs[l]).cuda())
    s.set_tree(np.asarray(tok).tolist(), np.asarray(parent).tolist())
    lg, codes, pred = traced_verify(s, shape, N)
    om = OM.Model(ow, L + N + 1, record=True)
    for l in range(shape.n_layers):
        om.K[l][:, :L] = ks[l]
        om.V[l][:, :L] = vs[l]
    ref = OS.tree_verify(om, L, tok, parent)
    fl = Flips(codes, om.record, shape, L, parent)
    ff = fl.check_first_flips()
    clean = [fl.row_clean(i) for i in range(N)]
    st, lo = check_rows(lg, ref, pred, clean)
    tally.add(st, lo, ff)
    return st, lo




def _torch():
    import torch
    return torch
