"""W4A8 matrix multiplication, by definition.

"GPU-Resident Speculative Decoding ...", Design > Small-Batch Verification
Kernels: int4 weights with one 16-bit scale per 32 inputs times int8
activations.  The product is

    y[t, n] = sum_g s_w[n, g] * s_a[t(, g)] * isum[t, n, g],
    isum[t, n, g] = sum_{k in group g} q_w[n, k] * q_a[t, k]   (exact integer)

The oracle evaluates it as the fp64 product of the dequantised operands (a
library matmul; every dequantised value is exact in fp64 and the fp64 rounding
error is far below the fp32 tolerance of the kernels).  ``group_sums`` computes
the integer part exactly (int64) for the bit-exact pins.
"""
from __future__ import annotations

import numpy as np

from .quant import GROUP, dequantize_act, dequantize_weights, unpack_q4


def w4a8_matmul(a_q, a_s, w_packed, w_s) -> np.ndarray:
    """(int8 [M][K], fp32 [M] or [M][K/32]) x (u32 [N][K/8], fp16 [N][K/32]) -> fp64 [M][N]."""
    wq = unpack_q4(w_packed)
    return dequantize_act(a_q, a_s) @ dequantize_weights(wq, w_s).T


def w4a8_matmul_codes(a_q, a_s, w_q, w_s) -> np.ndarray:
    """Same as ``w4a8_matmul`` with unpacked weight codes."""
    return dequantize_act(a_q, a_s) @ dequantize_weights(w_q, w_s).T


def group_sums(a_q, w_q) -> np.ndarray:
    """Exact integer group sums isum[t, n, g] (int64), brute force."""
    M, K = a_q.shape
    N = w_q.shape[0]
    a = a_q.astype(np.int64).reshape(M, 1, K // GROUP, GROUP)
    w = w_q.astype(np.int64).reshape(1, N, K // GROUP, GROUP)
    return (a * w).sum(axis=3)


def abs_terms(a_q, a_s, w_q, w_s) -> np.ndarray:
    """sum_g |s_w * s_a * isum| per (t, n): the scale of fp32 rounding error in y."""
    isum = np.abs(group_sums(a_q, w_q)).astype(np.float64)          # [M][N][G]
    sw = np.abs(w_s.astype(np.float64))[None, :, :]
    sa = np.abs(np.asarray(a_s, dtype=np.float64))
    if sa.ndim == 1:
        return (isum * sw).sum(axis=2) * sa[:, None]
    return (isum * sw * sa[:, None, :]).sum(axis=2)


def matvec_q4(w_packed, scales_f32, x) -> np.ndarray:
    """The blog's portable WGSL matvec ("WebGPU for LLM Inference, in depth", section
    "A quantised matrix-vector kernel in WGSL"), restated: y[row] = sum over packed
    words k and nibbles j of s[row, k/4] * (nibble - 8) * x[8k + j], with f32 scales
    and f32 activations (no activation quantisation).  Evaluated in fp64."""
    w_packed = np.asarray(w_packed, dtype=np.uint32)
    rows, words = w_packed.shape
    x = np.asarray(x, dtype=np.float64)
    y = np.zeros(rows, dtype=np.float64)
    for row in range(rows):
        acc = 0.0
        for k in range(words):
            s = float(scales_f32[row, k // 4])
            packed = int(w_packed[row, k])
            for j in range(8):
                q = float((packed >> (4 * j)) & 0xF) - 8.0
                acc += s * q * x[8 * k + j]
        y[row] = acc
    return y
