"""Building a library-held decoder from fp32 weights.

The offline converter of the pages (int4 codes with one fp16 scale per 32 inputs) runs
on the device through ``w4a8_quantize_weights``; ``fill(kind, layer, out)`` supplies the
fp32 weights of one tensor into a device buffer (e.g. from a checkpoint or a seeded
generator), one tensor at a time so that peak memory stays at one fp32 tensor.
"""
from __future__ import annotations

from . import (Model, T_DOWN, T_EMBED, T_GATE, T_K, T_LM_HEAD, T_O, T_Q, T_UP, T_V, w4a8_quantize_weights)


def tensor_dims(n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab):
    qd, kvd = n_heads * head_dim, n_kv_heads * head_dim
    return {T_Q: (qd, hidden), T_K: (kvd, hidden), T_V: (kvd, hidden), T_O: (hidden, qd),
            T_GATE: (ffn, hidden), T_UP: (ffn, hidden), T_DOWN: (hidden, ffn),
            T_EMBED: (vocab, hidden), T_LM_HEAD: (vocab, hidden)}


def build_model(n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab, tied, fill, rms_eps=1e-6,
                rope_base=10000.0, device="cuda"):
    import torch
    m = Model(n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab, tied, rms_eps, rope_base)
    dims = tensor_dims(n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab)
    kinds = [(k, l) for l in range(n_layers) for k in (T_Q, T_K, T_V, T_O, T_GATE, T_UP, T_DOWN)]
    kinds.append((T_EMBED, 0))
    if not tied:
        kinds.append((T_LM_HEAD, 0))
    for kind, layer in kinds:
        rows, cols = dims[kind]
        w = torch.empty((rows, cols), dtype=torch.float32, device=device)
        fill(kind, layer, w)
        wq, ws = w4a8_quantize_weights(w)
        m.load_tensor(kind, layer, wq, ws)
        torch.cuda.current_stream().synchronize()
        del w, wq, ws
    return m
