"""C-ABI library: builds, loads, exports every declared symbol, validates on the host (CPU only).

No compute call is made here: tfl_create is only given shapes that fail
validation before any device work.
"""
import ctypes
import os
import re

import pytest

import attention_qkv_gemm_gb300 as pkg
from attention_qkv_gemm_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return pkg.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "tfl.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tfl_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("tfl_create", "tfl_forward", "tfl_destroy", "tfl_status", "tfl_last_error", "tfl_forward_bf16",
              "tfl_forward_host", "tfl_forward_noalloc"):
        assert n in names
    assert set(pkg.EXPORTS) == set(names)


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_default_options(lib):
    o = pkg.tfl_default_options()
    assert o.precision == 2 and abs(o.ln_eps - 1e-5) < 1e-12
    assert o.wait_timeout_ns == 2_000_000_000 and o.use_graph == 1 and o.max_workspace_bytes == 0
    assert o.whole_stack == 1


def test_workspace_bytes(lib):
    s = pkg.TflShape(64, 1024, 128, 4, 512, 4, 0)
    M = 64 * 1024
    # h32, normed hi/lo, qkv, attention output, GELU output hi/lo (default precision 2)
    expect = M * 128 * 4 + 2 * M * 128 * 2 + M * 384 * 2 + M * 128 * 2 + 2 * M * 512 * 2
    got = pkg.tfl_workspace_bytes(s)
    assert expect <= got <= expect + 8 * 1024
    assert pkg.tfl_workspace_bytes(pkg.TflShape(1, 1, 100, 4, 512, 1, 0)) == 0


@pytest.mark.parametrize("shape,code", [
    ((1, 128, 128, 3, 512, 1, 0), pkg.TFL_ERR_INVALID_ARG),    # n_heads does not divide d_model
    ((1, 128, 128, 8, 512, 1, 0), pkg.TFL_ERR_UNSUPPORTED),    # head_dim 16
    ((1, 128, 192, 3, 512, 1, 0), pkg.TFL_ERR_UNSUPPORTED),    # d_model not 128 * 2^k
    ((1, 128, 128, 4, 500, 1, 0), pkg.TFL_ERR_UNSUPPORTED),    # d_ff not a multiple of 128
    ((0, 128, 128, 4, 512, 1, 0), pkg.TFL_ERR_INVALID_ARG),    # empty batch
    ((1, 128, 128, 4, 512, 1, 2), pkg.TFL_ERR_INVALID_ARG),    # bad norm placement
    ((1 << 16, 1 << 15, 128, 4, 512, 1, 0), pkg.TFL_ERR_UNSUPPORTED),  # B*S >= 2^31
])
def test_create_rejects_bad_shapes(lib, shape, code):
    s = pkg.TflShape(*shape)
    h = ctypes.c_void_p()
    w = pkg.TflWeights(None, shape[5], None, None)
    rc = lib.tfl_create(ctypes.byref(s), ctypes.byref(w), None, ctypes.byref(h))
    assert rc == code, pkg.tfl_last_error()
    assert h.value is None
    assert pkg.tfl_last_error() != ""


def test_null_arguments_are_rejected(lib):
    assert lib.tfl_forward(None, None, None, 1, None, None) == pkg.TFL_ERR_INVALID_ARG
    assert lib.tfl_status(None, None) == pkg.TFL_ERR_INVALID_ARG
    assert lib.tfl_create(None, None, None, None) == pkg.TFL_ERR_INVALID_ARG
    lib.tfl_destroy(None)  # no-op
