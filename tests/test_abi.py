"""The C-ABI library builds, loads and exports every symbol include/w4a8.h declares (CPU)."""
import ctypes
import os
import re

import numpy as np
import pytest

import w4a8_verify_gb300 as W
from w4a8_verify_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return W.lib()


def _header_symbols():
    txt = open(os.path.join(ROOT, "include", "w4a8.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[\w\*\s]+?\b(w4a8_\w+|tree_verify_step|accept_greedy|kv_compact|"
                       r"ngram_draft|spec_window|spec_poll)\s*\(", txt, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _header_symbols()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    # the binding declares exactly the header's functions
    assert sorted(W.declared_symbols()) == names


def test_status_strings_and_version(lib):
    assert W.status_str(0) == "ok"
    assert "shape" in W.status_str(2)
    assert lib.w4a8_abi_version() >= 1


def test_host_pack_matches_oracle(lib):
    from oracle import quant as Q
    rng = np.random.default_rng(0)
    q = rng.integers(-8, 8, size=(5, 64)).astype(np.int8)
    assert np.array_equal(W.w4a8_pack_weights(q), Q.pack_q4(q))
    bad = q.copy(); bad[0, 0] = 9
    with pytest.raises(W.W4A8Error):
        W.w4a8_pack_weights(bad)


def test_host_argument_checks_without_gpu(lib):
    sz = ctypes.c_size_t()
    assert lib.w4a8_matmul_workspace_bytes(17, 64, 32, ctypes.byref(sz)) == 2      # M > 16
    assert lib.w4a8_matmul_workspace_bytes(1, 48, 32, ctypes.byref(sz)) == 2      # K % 32
    assert lib.w4a8_matmul_workspace_bytes(1, 64, 24, ctypes.byref(sz)) == 2      # N % 16
    assert lib.w4a8_matmul(None, None, 1, 64, None, None, 32, None, None, 0, None) == 1
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.w4a8_weight_layout_bytes(32, 96, ctypes.byref(a), ctypes.byref(b)) == 0
    assert a.value == 2 * 2 * 128 * 4 and b.value == 2 * 2 * 32 * 2


def test_matmul_schedule_depends_on_shape_only(lib):
    for K, N in [(896, 4864), (4864, 896), (4096, 14336), (14336, 4096), (4096, 128256), (256, 512), (704, 256)]:
        S = W.w4a8_matmul_slices(K, N)
        assert 1 <= S <= max(1, (K + 63) // 64 // 2)


def test_model_shapes_the_tree_attention_cannot_hold_are_rejected(lib):
    """Head size 128 with more than 4 query heads per KV head needs more than a block's shared
    memory in the 16-node tree attention: model creation says so (W4A8_ERR_SHAPE) before any
    device allocation; the benchmarked grouping (4 per KV head at 128, 7 at 64) stays valid."""
    def create(n_heads, n_kv_heads, head_dim):
        d = W.ModelDesc(1, 512, n_heads, n_kv_heads, head_dim, 1024, 4096, 0, 1e-6, 10000.0)
        h = ctypes.c_void_p()
        st = lib.w4a8_model_create(ctypes.byref(d), ctypes.byref(h))
        if st == 0:
            lib.w4a8_model_destroy(h)
        return st
    assert create(40, 8, 128) == 2         # 5 per KV head at 128
    assert create(28, 4, 128) == 2         # 7 per KV head at 128
    assert create(64, 8, 128) == 2         # 8 per KV head at 128
    assert create(8, 1, 64) != 2           # 8 per KV head at 64 fits
    assert create(32, 8, 128) != 2         # 4 per KV head at 128 fits
