"""Quantisers and the packed int4 layout.

* Weight format: 4-bit codes with one 16-bit scale per 32 inputs ("GPU-Resident
  Speculative Decoding ...", Design > Small-Batch Verification Kernels;
  Implementation: offline converter).
* Packed layout: eight codes per u32, code j of word k is element 8k+j in bits
  4j..4j+3, stored as 0..15 meaning -8..7 ("WebGPU for LLM Inference, in depth",
  section "A quantised matrix-vector kernel in WGSL").
* Activations: int8 codes; per token (default) or per block of 32 values
  ("GPU-Resident Speculative Decoding ...", Design > Small-Batch Verification
  Kernels says per block of 32; the per-token absmax reading is the default).

Readings where the pages are silent:
* weight scale s = fp16(fp32(absmax) / 7), code q = clamp(rint(w / s), -8, 7)
  with rint = round half to even, taken in fp32; absmax = 0 (or s rounding to
  0) gives s = 0 and q = 0.
* activation scale s = fp32(absmax) / 127 (IEEE fp32 division), code
  q = clamp(rint(x / s), -127, 127) in fp32; absmax = 0 gives s = 0, q = 0.
"""
from __future__ import annotations

import numpy as np

GROUP = 32


def quantize_weights_g32(w: np.ndarray):
    """fp32 [N][K] -> (int8 codes [N][K], fp16 scales [N][K/32])."""
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    assert K % GROUP == 0
    g = w.reshape(N, K // GROUP, GROUP)
    amax = np.abs(g).max(axis=2)                                   # exact in fp32
    s16 = (amax / np.float32(7.0)).astype(np.float32).astype(np.float16)
    s32 = s16.astype(np.float32)
    safe = np.where(s32 > 0, s32, np.float32(1.0))
    q = np.rint((g / safe[:, :, None]).astype(np.float32))
    q = np.clip(q, -8, 7)
    q = np.where((s32 > 0)[:, :, None], q, 0).astype(np.int8)
    s16 = np.where(s32 > 0, s16, np.float16(0.0)).astype(np.float16)
    return q.reshape(N, K), s16


def pack_q4(q: np.ndarray) -> np.ndarray:
    """int8 codes [N][K] in [-8,7] -> u32 [N][K/8], nibble j of word k = element 8k+j, value q+8."""
    q = np.asarray(q)
    N, K = q.shape
    assert K % 8 == 0
    assert q.min() >= -8 and q.max() <= 7
    nib = (q.astype(np.int32) + 8).astype(np.uint32).reshape(N, K // 8, 8)
    out = np.zeros((N, K // 8), dtype=np.uint32)
    for j in range(8):
        out |= nib[:, :, j] << np.uint32(4 * j)
    return out


def unpack_q4(w: np.ndarray) -> np.ndarray:
    """u32 [N][K/8] -> int8 codes [N][K]."""
    w = np.asarray(w, dtype=np.uint32)
    N, W = w.shape
    out = np.empty((N, W, 8), dtype=np.int8)
    for j in range(8):
        out[:, :, j] = ((w >> np.uint32(4 * j)) & np.uint32(15)).astype(np.int16) - 8
    return out.reshape(N, W * 8)


def dequantize_weights(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Codes and fp16 group scales -> fp64 weights s_g * q_k (exact)."""
    N, K = q.shape
    return (q.astype(np.float64).reshape(N, K // GROUP, GROUP)
            * s.astype(np.float64)[:, :, None]).reshape(N, K)


def quantize_act_per_token(x: np.ndarray):
    """fp32 [M][K] -> (int8 [M][K], fp32 scale [M]).  Decision taken in fp32."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=1)
    s = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    q = np.rint((x / safe[:, None]).astype(np.float32))
    q = np.clip(q, -127, 127)
    q = np.where((s > 0)[:, None], q, 0).astype(np.int8)
    return q, s


def quantize_act_per_block32(x: np.ndarray):
    """fp32 [M][K] -> (int8 [M][K], fp32 scale [M][K/32]): the same rule per block of 32."""
    x = np.asarray(x, dtype=np.float32)
    M, K = x.shape
    assert K % GROUP == 0
    q, s = quantize_act_per_token(x.reshape(M * (K // GROUP), GROUP))
    return q.reshape(M, K), s.reshape(M, K // GROUP)


def dequantize_act(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    q = q.astype(np.float64)
    s = np.asarray(s, dtype=np.float64)
    if s.ndim == 1:
        return q * s[:, None]
    M, K = q.shape
    return (q.reshape(M, K // GROUP, GROUP) * s[:, :, None]).reshape(M, K)
