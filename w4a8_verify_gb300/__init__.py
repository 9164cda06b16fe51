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
_u16, _u32, _dbl = _c.c_uint16, _c.c_uint32, _c.c_double


class ModelDesc(_c.Structure):
    _fields_ = [("n_layers", _i32), ("hidden", _i32), ("n_heads", _i32), ("n_kv_heads", _i32), ("head_dim", _i32),
                ("ffn", _i32), ("vocab", _i32), ("tied", _i32), ("rms_eps", _f32), ("rope_base", _f32)]


class SessionDesc(_c.Structure):
    _fields_ = [("kv_cap", _i32), ("ctx_cap", _i32), ("max_window", _i32), ("eos_id", _i32), ("mem_cap", _i32)]


class Ctl(_c.Structure):
    _fields_ = [("committed_len", _u32), ("ctx_len", _u32), ("n_valid", _u32), ("root_tok", _i32),
                ("n_generated", _u32), ("max_new", _u32), ("flags", _u32), ("step_idx", _u32)]


class Ctl16(_c.Structure):
    _fields_ = [("committed_len", _u32), ("n_generated", _u32), ("flags", _u32), ("root_tok", _i32)]


class StepStats(_c.Structure):
    _fields_ = [("n_accepted_drafts", _u16), ("best_match_len", _u16), ("n_nodes", _u16), ("n_emitted", _u16),
                ("t_lo", _u32)]


class DecodeOpts(_c.Structure):
    _fields_ = [("max_new", _i32), ("window", _i32), ("fixed_width", _i32), ("in_flight", _i32),
                ("timeout_us", _i64), ("n_widths", _i32), ("widths", _i32 * 8), ("t_us", _f32 * 8)]


class DecodeReport(_c.Structure):
    _fields_ = [("n_tokens", _i32), ("n_steps", _i32), ("n_windows", _i32), ("host_syncs", _i32),
                ("accepted_drafts", _i32), ("width_steps", _i32 * 17), ("flags", _u32), ("device_us", _dbl),
                ("kernels", _i64)]


FLAG_TERMINATED, FLAG_ERR_CAPACITY, FLAG_ERR_TOKEN, FLAG_ERR_TREE, FLAG_ERR_TIMEOUT = 1, 2, 4, 8, 16
T_Q, T_K, T_V, T_O, T_GATE, T_UP, T_DOWN, T_EMBED, T_LM_HEAD = range(9)

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
    "w4a8_matmul_inject_timeout": [_vp, _vp, _i32, _i32, _vp, _vp, _i32, _vp, _vp, _sz, _vp],
    "w4a8_matmul_nondet": [_vp, _vp, _i32, _i32, _vp, _vp, _i32, _vp, _vp, _sz, _vp],
    "w4a8_matmul_per32": [_vp, _vp, _i32, _i32, _vp, _vp, _i32, _vp, _vp, _sz, _vp],
    "w4a8_matmul_check": [_vp, _i32, _i32, _i32, _c.POINTER(_c.c_uint32)],
    "w4a8_matmul_noalloc": [_vp, _vp, _i32, _i32, _vp, _vp, _i32, _vp, _vp],
    "w4a8_matmul_noalloc_check": [_c.POINTER(_c.c_uint32)],
    "w4a8_model_create": [_c.POINTER(ModelDesc), _c.POINTER(_vp)],
    "w4a8_model_load_tensor": [_vp, _i32, _i32, _vp, _vp, _vp],
    "w4a8_model_weight_bytes": [_vp, _c.POINTER(_sz)],
    "w4a8_model_destroy": [_vp],
    "w4a8_session_create": [_vp, _c.POINTER(SessionDesc), _c.POINTER(_vp)],
    "w4a8_session_destroy": [_vp],
    "w4a8_prefill": [_vp, _vp, _i32, _i32, _vp],
    "tree_verify_step": [_vp, _i32, _vp, _vp],
    "w4a8_model_trace_bytes": [_vp, _i32, _c.POINTER(_sz)],
    "w4a8_tree_verify_trace": [_vp, _i32, _vp, _vp, _sz, _vp],
    "accept_greedy": [_vp, _i32, _vp],
    "kv_compact": [_vp, _vp],
    "ngram_draft": [_vp, _vp],
    "w4a8_spec_step": [_vp, _i32, _vp],
    "spec_window": [_vp, _i32, _i32, _vp],
    "spec_poll": [_vp, _c.POINTER(Ctl16), _c.POINTER(StepStats), _c.POINTER(_i32), _c.POINTER(_i32),
                  _c.POINTER(_i32), _i64],
    "w4a8_calibrate": [_vp, _c.POINTER(_i32), _i32, _i32, _i32, _c.POINTER(_f32)],
    "w4a8_decode": [_vp, _c.POINTER(_i32), _i32, _c.POINTER(DecodeOpts), _c.POINTER(_i32), _c.POINTER(_i32),
                    _c.POINTER(DecodeReport), _vp],
    "w4a8_generate": [_vp, _c.POINTER(DecodeOpts), _c.POINTER(_i32), _c.POINTER(_i32), _c.POINTER(DecodeReport),
                      _vp],
    "w4a8_time_matmuls": [_vp, _i32, _i32, _c.POINTER(_dbl), _c.POINTER(_dbl), _c.POINTER(_i32)],
    "w4a8_session_get_ctl": [_vp, _c.POINTER(Ctl)],
    "w4a8_session_raise_flags": [_vp, _u32, _vp],
    "w4a8_session_set_tree": [_vp, _c.POINTER(_i32), _c.POINTER(_i32), _i32],
    "w4a8_session_get_tree": [_vp, _c.POINTER(_i32), _c.POINTER(_i32), _c.POINTER(_i32), _c.POINTER(_i32),
                              _c.POINTER(_i32)],
    "w4a8_session_get_pred": [_vp, _c.POINTER(_i32), _i32],
    "w4a8_session_get_context": [_vp, _c.POINTER(_i32), _i32, _c.POINTER(_i32)],
    "w4a8_session_copy_kv": [_vp, _i32, _i32, _i32, _vp, _vp, _vp],
    "w4a8_session_load_kv": [_vp, _i32, _i32, _i32, _vp, _vp, _vp],
    "w4a8_session_attention": [_vp, _i32, _i32, _vp, _vp, _vp],
    "w4a8_session_memory_append": [_vp, _c.POINTER(_i32), _i32],
    "w4a8_session_memory_clear": [_vp],
    "w4a8_session_memory_get": [_vp, _c.POINTER(_i32), _i32, _c.POINTER(_i32)],
    "w4a8_controller_create": [_c.POINTER(_i32), _c.POINTER(_f32), _i32, _c.POINTER(_vp)],
    "w4a8_controller_destroy": [_vp],
    "w4a8_controller_choose": [_vp],
    "w4a8_controller_observe": [_vp, _i32, _c.POINTER(StepStats), _i32, _dbl],
    "w4a8_controller_expected_tokens": [_vp, _i32],
    "w4a8_controller_cost": [_vp, _i32],
}
_RESTYPE = {"w4a8_status_str": _c.c_char_p, "w4a8_model_destroy": None, "w4a8_session_destroy": None,
            "w4a8_controller_destroy": None, "w4a8_controller_expected_tokens": _dbl, "w4a8_controller_cost": _dbl}


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


def w4a8_matmul_check(workspace, M, K, N):
    """Device status word of a matmul workspace (0 = every bounded wait completed)."""
    f = _c.c_uint32()
    st = lib().w4a8_matmul_check(_ptr(workspace), M, K, N, _c.byref(f))
    if st not in (0, 7):
        raise W4A8Error("w4a8_matmul_check", st)
    return f.value


def w4a8_matmul_noalloc(a_q, a_s, w_t, s_t, N, y, stream=None):
    """w4a8_matmul with the library's own static scratch (no allocation; y is caller-owned)."""
    M, K = a_q.shape
    _call("w4a8_matmul_noalloc", _ptr(a_q), _ptr(a_s), M, K, _ptr(w_t), _ptr(s_t), N, _ptr(y), _stream(stream))
    return y


def w4a8_matmul_per32(a_q, a_s, w_t, s_t, N, y=None, workspace=None, stream=None):
    """W4A8 product with per-32 activation scales a_s [M][K/32] (w4a8_matmul_per32)."""
    import torch
    M, K = a_q.shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=a_q.device)
    need = w4a8_matmul_workspace_bytes(M, K, N)
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=a_q.device)
    _call("w4a8_matmul_per32", _ptr(a_q), _ptr(a_s), M, K, _ptr(w_t), _ptr(s_t), N, _ptr(y), _ptr(workspace),
          workspace.numel() * workspace.element_size(), _stream(stream))
    return y


def w4a8_matmul_nondet(a_q, a_s, w_t, s_t, N, y=None, workspace=None, stream=None):
    """The non-deterministic fast variant (slices combined with float atomics)."""
    import torch
    M, K = a_q.shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=a_q.device)
    need = w4a8_matmul_workspace_bytes(M, K, N)
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=a_q.device)
    _call("w4a8_matmul_nondet", _ptr(a_q), _ptr(a_s), M, K, _ptr(w_t), _ptr(s_t), N, _ptr(y), _ptr(workspace),
          workspace.numel() * workspace.element_size(), _stream(stream))
    return y


def w4a8_matmul_inject_timeout(a_q, a_s, w_t, s_t, N, y, workspace, stream=None):
    """Test-only: the matmul with a copy warp that issues nothing, so that its bounded waits
    expire and the workspace status word reports the timeout (w4a8_matmul_inject_timeout)."""
    M, K = a_q.shape
    _call("w4a8_matmul_inject_timeout", _ptr(a_q), _ptr(a_s), M, K, _ptr(w_t), _ptr(s_t), N, _ptr(y),
          _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))


def w4a8_matmul_noalloc_check():
    """Status word of the last w4a8_matmul_noalloc call on the current device (0 = every
    bounded wait completed; synchronous: call after that stream has finished)."""
    f = _c.c_uint32()
    st = lib().w4a8_matmul_noalloc_check(_c.byref(f))
    if st not in (0, 7):
        raise W4A8Error("w4a8_matmul_noalloc_check", st)
    return f.value


def w4a8_matmul(a_q, a_s, w_t, s_t, N, y=None, workspace=None, stream=None):
    import torch
    M, K = a_q.shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=a_q.device)
    need = w4a8_matmul_workspace_bytes(M, K, N)
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=a_q.device)
    _call("w4a8_matmul", _ptr(a_q), _ptr(a_s), M, K, _ptr(w_t), _ptr(s_t), N, _ptr(y), _ptr(workspace),
          workspace.numel() * workspace.element_size(), _stream(stream))
    return y


# ------------------------------------------------------------------------ model/session

def _arr(vals, ctype=_i32):
    vals = list(vals)
    return (ctype * max(1, len(vals)))(*vals)


class Model:
    """A decoder held by the library (w4a8_model)."""

    def __init__(self, n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab, tied,
                 rms_eps=1e-6, rope_base=10000.0):
        self.desc = ModelDesc(n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab, int(bool(tied)),
                              rms_eps, rope_base)
        h = _vp()
        _call("w4a8_model_create", _c.byref(self.desc), _c.byref(h))
        self.h = h

    def load_tensor(self, kind, layer, w_p2, s_p2, stream=None):
        _call("w4a8_model_load_tensor", self.h, int(kind), int(layer), _ptr(w_p2), _ptr(s_p2), _stream(stream))

    def weight_bytes(self):
        b = _sz()
        _call("w4a8_model_weight_bytes", self.h, _c.byref(b))
        return b.value

    def close(self):
        if getattr(self, "h", None):
            lib().w4a8_model_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Session:
    """A decoding session (w4a8_session) on a Model."""

    def __init__(self, model, kv_cap, ctx_cap, max_window=16, eos_id=-1, mem_cap=0):
        self.model = model
        self.desc = SessionDesc(kv_cap, ctx_cap, max_window, eos_id, mem_cap)
        h = _vp()
        _call("w4a8_session_create", model.h, _c.byref(self.desc), _c.byref(h))
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            lib().w4a8_session_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # device-side operations (asynchronous on the current stream)
    def prefill(self, prompt_dev, max_new, stream=None):
        _call("w4a8_prefill", self.h, _ptr(prompt_dev), int(prompt_dev.numel()), int(max_new), _stream(stream))

    def tree_verify_step(self, N, logits=None, stream=None):
        _call("tree_verify_step", self.h, int(N), _ptr(logits), _stream(stream))

    def trace_bytes(self, N):
        n = _sz()
        _call("w4a8_model_trace_bytes", self.model.h, int(N), _c.byref(n))
        return n.value

    def tree_verify_trace(self, N, codes, logits=None, stream=None):
        """tree_verify_step that also writes the int8 codes of every quantisation point into
        the device int8 buffer ``codes`` (w4a8_tree_verify_trace)."""
        _call("w4a8_tree_verify_trace", self.h, int(N), _ptr(logits), _ptr(codes),
              codes.numel() * codes.element_size(), _stream(stream))

    def accept_greedy(self, N, stream=None):
        _call("accept_greedy", self.h, int(N), _stream(stream))

    def kv_compact(self, stream=None):
        _call("kv_compact", self.h, _stream(stream))

    def ngram_draft(self, stream=None):
        _call("ngram_draft", self.h, _stream(stream))

    def spec_step(self, N, stream=None):
        _call("w4a8_spec_step", self.h, int(N), _stream(stream))

    def spec_window(self, N, W, stream=None):
        _call("spec_window", self.h, int(N), int(W), _stream(stream))

    def spec_poll(self, W, timeout_us=-1):
        c = Ctl16()
        st = (StepStats * max(1, W))()
        toks = (_i32 * (16 * max(1, W)))()
        ns, nt = _i32(), _i32()
        _call("spec_poll", self.h, _c.byref(c), st, _c.byref(ns), toks, _c.byref(nt), int(timeout_us))
        return c, list(st)[:ns.value], list(toks)[:nt.value]

    def calibrate(self, widths, reps=20, trials=5):
        out = (_f32 * len(widths))()
        _call("w4a8_calibrate", self.h, _arr(widths), len(widths), int(reps), int(trials), out)
        return list(out)

    @staticmethod
    def _opts(max_new, window, fixed_width, in_flight, widths, t_us, timeout_us):
        o = DecodeOpts()
        o.max_new, o.window, o.fixed_width, o.in_flight, o.timeout_us = max_new, window, fixed_width, in_flight, timeout_us
        o.n_widths = len(widths)
        for i, (w, t) in enumerate(zip(widths, t_us)):
            o.widths[i], o.t_us[i] = int(w), float(t)
        return o

    def generate(self, max_new, window=4, fixed_width=0, in_flight=2, widths=(), t_us=(), timeout_us=-1,
                 stream=None):
        """Window loop on a prefilled session; returns (tokens, DecodeReport)."""
        o = self._opts(max_new, window, fixed_width, in_flight, widths, t_us, timeout_us)
        out = (_i32 * max(1, max_new))()
        n_out = _i32()
        rep = DecodeReport()
        _call("w4a8_generate", self.h, _c.byref(o), out, _c.byref(n_out), _c.byref(rep), _stream(stream))
        return list(out)[:n_out.value], rep

    def time_matmuls(self, N, reps=5):
        us, by, nl = _dbl(), _dbl(), _i32()
        _call("w4a8_time_matmuls", self.h, int(N), int(reps), _c.byref(us), _c.byref(by), _c.byref(nl))
        return us.value, by.value, nl.value

    def decode(self, prompt, max_new, window=4, fixed_width=0, in_flight=2, widths=(), t_us=(),
               timeout_us=-1, stream=None):
        """End-to-end decode from a host prompt; returns (tokens, DecodeReport)."""
        o = DecodeOpts()
        o.max_new, o.window, o.fixed_width, o.in_flight, o.timeout_us = max_new, window, fixed_width, in_flight, timeout_us
        o.n_widths = len(widths)
        for i, (w, t) in enumerate(zip(widths, t_us)):
            o.widths[i], o.t_us[i] = int(w), float(t)
        p = _arr([int(t) for t in prompt])
        out = (_i32 * max(1, max_new))()
        n_out = _i32()
        rep = DecodeReport()
        _call("w4a8_decode", self.h, p, len(prompt), _c.byref(o), out, _c.byref(n_out), _c.byref(rep),
              _stream(stream))
        return list(out)[:n_out.value], rep

    def raise_flags(self, flags, stream=None):
        _call("w4a8_session_raise_flags", self.h, int(flags), _stream(stream))

    # synchronous state access
    def ctl(self):
        c = Ctl()
        _call("w4a8_session_get_ctl", self.h, _c.byref(c))
        return c

    def set_tree(self, tok, parent):
        n = len(tok)
        _call("w4a8_session_set_tree", self.h, _arr(tok), _arr(parent), n)

    def tree(self):
        tok, par, dep = (_i32 * 16)(), (_i32 * 16)(), (_i32 * 16)()
        nv, bl = _i32(), _i32()
        _call("w4a8_session_get_tree", self.h, tok, par, dep, _c.byref(nv), _c.byref(bl))
        return list(tok), list(par), list(dep), nv.value, bl.value

    def pred(self, n):
        out = (_i32 * n)()
        _call("w4a8_session_get_pred", self.h, out, int(n))
        return list(out)

    def context(self, cap=1 << 16):
        out = (_i32 * cap)()
        n = _i32()
        _call("w4a8_session_get_context", self.h, out, cap, _c.byref(n))
        return list(out)[:min(cap, n.value)]

    def copy_kv(self, layer, slot0, n, k_out, v_out, stream=None):
        _call("w4a8_session_copy_kv", self.h, int(layer), int(slot0), int(n), _ptr(k_out), _ptr(v_out),
              _stream(stream))

    def memory_append(self, tokens):
        """Appends an earlier output to the session memory (w4a8_session_memory_append)."""
        _call("w4a8_session_memory_append", self.h, _arr([int(t) for t in tokens]), len(tokens))

    def memory_clear(self):
        _call("w4a8_session_memory_clear", self.h)

    def memory(self, cap=1 << 16):
        out = (_i32 * cap)()
        n = _i32()
        _call("w4a8_session_memory_get", self.h, out, cap, _c.byref(n))
        return list(out)[:min(cap, n.value)]

    def load_kv(self, layer, slot0, n, k_in, v_in, stream=None):
        _call("w4a8_session_load_kv", self.h, int(layer), int(slot0), int(n), _ptr(k_in), _ptr(v_in),
              _stream(stream))

    def attention(self, layer, n, q, out, stream=None):
        """Tree attention of one layer for device queries q [n][n_heads][head_dim] (after RoPE
        and the 1/sqrt(head_dim) scale) into out [n][n_heads * head_dim] (w4a8_session_attention)."""
        _call("w4a8_session_attention", self.h, int(layer), int(n), _ptr(q), _ptr(out), _stream(stream))


class Controller:
    """The host width controller (w4a8_controller)."""

    def __init__(self, widths, t_us):
        h = _vp()
        _call("w4a8_controller_create", _arr(widths), _arr(t_us, _f32), len(widths), _c.byref(h))
        self.h = h

    def choose(self):
        return lib().w4a8_controller_choose(self.h)

    def observe(self, width, stats, interval_us=0.0):
        arr = (StepStats * max(1, len(stats)))()
        for i, st in enumerate(stats):
            arr[i] = st if isinstance(st, StepStats) else StepStats(*st)
        _call("w4a8_controller_observe", self.h, int(width), arr, len(stats), float(interval_us))

    def expected_tokens(self, width):
        return lib().w4a8_controller_expected_tokens(self.h, int(width))

    def cost(self, width):
        return lib().w4a8_controller_cost(self.h, int(width))

    def __del__(self):
        try:
            if getattr(self, "h", None):
                lib().w4a8_controller_destroy(self.h)
                self.h = None
        except Exception:
            pass
