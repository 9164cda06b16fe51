"""ctypes binding and build of ``libsynth.so`` (the device copy of gen.py's streams).

The host side computes the stream key and the fp32 constants exactly as gen.py does
and passes them in, so both sides draw identical values."""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import gen

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "libsynth.so")
_lib = None


def build() -> str:
    src = os.path.join(HERE, "synth.cu")
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(src):
        cmd = [os.environ.get("NVCC", "nvcc"), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
               "-Xcompiler", "-fPIC,-fvisibility=hidden", "-shared", src, "-o", LIB]
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        if r.returncode != 0:
            raise RuntimeError(r.stdout)
    return LIB


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError("libsynth.so is not built: run __graft_entry__.build()")
        L = ctypes.CDLL(LIB)
        u64, vp, f32, i32, i64 = ctypes.c_uint64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int, ctypes.c_longlong
        L.synth_normal.argtypes = [u64, u64, u64, f32, vp, vp]
        L.synth_dense.argtypes = [u64, i32, i32, i32, i64, i64, f32, vp, vp]
        L.synth_codes.argtypes = [u64, u64, u64, vp, vp]
        L.synth_scales.argtypes = [u64, u64, u64, f32, f32, vp, vp]
        for f in (L.synth_normal, L.synth_dense, L.synth_codes, L.synth_scales):
            f.restype = ctypes.c_int
        _lib = L
    return _lib


def _stream(stream):
    return ctypes.c_void_p(stream) if stream else None


def _check(rc):
    if rc != 0:
        raise RuntimeError("synth kernel launch failed with CUDA error %d" % rc)


def normal(seed, stream_id, start, out, sigma, stream=0):
    """Fill device fp32 tensor ``out`` (numel n) with gen.normal(seed, stream_id, start, n, sigma)."""
    _check(lib().synth_normal(gen.stream_key(seed, stream_id), start, out.numel(),
                              float(gen.sigma_mult(sigma)), out.data_ptr(), _stream(stream)))


def dense_weight(shape, seed, stream_id, rows, cols, real_rows, real_cols, out, row0=0, stream=0):
    """Device fp32 rows [row0, row0+out.shape[0]) of gen.dense_weight."""
    _check(lib().synth_dense(gen.stream_key(seed, stream_id), cols, real_rows, real_cols, row0, out.shape[0],
                             float(gen.sigma_mult(shape.weight_sigma)), out.data_ptr(), _stream(stream)))


def uniform_codes(seed, stream_id, start, out, stream=0):
    _check(lib().synth_codes(gen.stream_key(seed, stream_id), start, out.numel(), out.data_ptr(), _stream(stream)))


def uniform_scales(seed, stream_id, start, out, lo=0.001, hi=0.02, stream=0):
    """Device fp16 tensor (stored as int16/uint16 bits) of gen.uniform_scales."""
    _check(lib().synth_scales(gen.stream_key(seed, stream_id), start, out.numel(), float(np.float32(hi - lo)),
                              float(np.float32(lo)), out.data_ptr(), _stream(stream)))
