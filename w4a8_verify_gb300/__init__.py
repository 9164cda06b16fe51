"""Python binding of ``libw4a8.so`` (the sm_103a library declared in include/w4a8.h).

Argument marshalling only: every function forwards torch tensors' device pointers
and the current CUDA stream to the C ABI function of the same name and raises on a
non-zero status.  The library must be built (``__graft_entry__.build()``); there is
no fallback path.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libw4a8.so")

_lib = None

_c = ctypes
_vp, _i32, _u64, _sz, _f32, _i64 = _c.c_void_p, _c.c_int, _c.c_uint64, _c.c_size_t, _c.c_float, _c.c_int64

# name -> argtypes (restype int = w4a8_status unless listed in _RESTYPE)
_SIGNATURES = {
    "w4a8_status_str": [_i32],
    "w4a8_abi_version": [],
    "w4a8_pack_weights": [_vp, _i32, _i32, _vp],
    "w4a8_quantize_weights": [_vp, _i32, _i32, _vp, _vp, _vp],
    "w4a8_weight_layout_bytes": [_i32, _i32, _c.POINTER(_sz), _c.POINTER(_sz)],
    "w4a8_repack_weights": [_vp, _vp, _i32, _i32, _vp, _vp, _vp],
    "w4a8_quantize_rows": [_vp, _i32, _i32, _i32, _vp, _vp, _vp],
    "w4a8_matmul_workspace_bytes": [_i32, _i32, _i32, _c.POINTER(_sz)],
    "w4a8_matmul": [_vp, _vp, _i32, _i32, _vp, _vp, _i32, _vp, _vp, _sz, _vp],
    "w4a8_matmul_slices": [_i32, _i32],
}
_RESTYPE = {"w4a8_status_str": _c.c_char_p}


class W4A8Error(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (fn, status_str(status), status))


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libw4a8.so not found at %s: run __graft_entry__.build()" % LIB_PATH)
        L = _c.CDLL(LIB_PATH)
        for name, args in _SIGNATURES.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = _RESTYPE.get(name, _c.c_int)
        _lib = L
    return _lib


def declared_symbols():
    return list(_SIGNATURES)


def status_str(s: int) -> str:
    return lib().w4a8_status_str(int(s)).decode()


def _call(name, *args):
    st = getattr(lib(), name)(*args)
    if st != 0:
        raise W4A8Error(name, st)
    return st


def _ptr(t):
    return None if t is None else _c.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return _c.c_void_p(s.cuda_stream)


# ----------------------------------------------------------------------------- weights

def w4a8_pack_weights(q):
    """int8 codes (host numpy [N][K]) -> packed u32 words (host numpy [N][K/8])."""
    import numpy as np
    q = np.ascontiguousarray(q, dtype=np.int8)
    N, K = q.shape
    out = np.empty((N, K // 8), dtype=np.uint32)
    _call("w4a8_pack_weights", q.ctypes.data_as(_vp), N, K, out.ctypes.data_as(_vp))
    return out


def w4a8_quantize_weights(w, w_p2=None, s_p2=None, stream=None):
    """fp32 device [N][K] -> (int32-viewed u32 words [N][K/8], int16-viewed fp16 scales [N][K/32])."""
    import torch
    N, K = w.shape
    if w_p2 is None:
        w_p2 = torch.empty((N, K // 8), dtype=torch.int32, device=w.device)
    if s_p2 is None:
        s_p2 = torch.empty((N, K // 32), dtype=torch.int16, device=w.device)
    _call("w4a8_quantize_weights", _ptr(w), N, K, _ptr(w_p2), _ptr(s_p2), _stream(stream))
    return w_p2, s_p2


def w4a8_weight_layout_bytes(N, K):
    wb, sb = _sz(), _sz()
    _call("w4a8_weight_layout_bytes", N, K, _c.byref(wb), _c.byref(sb))
    return wb.value, sb.value


def w4a8_repack_weights(w_p2, s_p2, N, K, stream=None):
    """P2 layout -> tiled layout (device tensors, int32 words / int16 scales)."""
    import torch
    wb, sb = w4a8_weight_layout_bytes(N, K)
    w_t = torch.empty(wb // 4, dtype=torch.int32, device=w_p2.device)
    s_t = torch.empty(sb // 2, dtype=torch.int16, device=w_p2.device)
    _call("w4a8_repack_weights", _ptr(w_p2), _ptr(s_p2), N, K, _ptr(w_t), _ptr(s_t), _stream(stream))
    return w_t, s_t


# ------------------------------------------------------------------------- activations

def w4a8_quantize_rows(x, mode=0, stream=None):
    import torch
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    s = torch.empty((M,) if mode == 0 else (M, K // 32), dtype=torch.float32, device=x.device)
    _call("w4a8_quantize_rows", _ptr(x), M, K, int(mode), _ptr(q), _ptr(s), _stream(stream))
    return q, s


# ------------------------------------------------------------------------------ matmul

def w4a8_matmul_workspace_bytes(M, K, N):
    b = _sz()
    _call("w4a8_matmul_workspace_bytes", M, K, N, _c.byref(b))
    return b.value


def w4a8_matmul_slices(K, N):
    return lib().w4a8_matmul_slices(K, N)


def w4a8_matmul(a_q, a_s, w_t, s_t, N, y=None, workspace=None, stream=None):
    import torch
    M, K = a_q.shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=a_q.device)
    need = w4a8_matmul_workspace_bytes(M, K, N)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=a_q.device)
    _call("w4a8_matmul", _ptr(a_q), _ptr(a_s), M, K, _ptr(w_t), _ptr(s_t), N, _ptr(y), _ptr(workspace),
          workspace.numel() * workspace.element_size(), _stream(stream))
    return y
