"""Python binding of ``libtfl.so``, the GB300 (sm_103a) Transformer-stack forward.

Argument marshalling only: every step of the forward runs in the library's
CUDA kernels.  The functions mirror the C ABI in ``include/tfl.h``
(``tfl_create``, ``tfl_forward``, ``tfl_forward_host``, ``tfl_status``,
``tfl_destroy``, ...).  ``TransformerStack`` is a small convenience wrapper
that keeps torch device tensors for the caller.

Loading fails loudly (``ImportError`` from ``load()``) when the library has
not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtfl.so")

TFL_OK = 0
TFL_ERR_INVALID_ARG = -1
TFL_ERR_UNSUPPORTED = -2
TFL_ERR_OOM = -3
TFL_ERR_CUDA = -4
TFL_ERR_DEVICE_TIMEOUT = -5
TFL_ERR_BAD_LENGTHS = -6

KIND_NAMES = {1: "rownorm", 2: "gemm_qkv", 3: "attention", 4: "gemm_oproj", 5: "gemm_ffn1", 6: "gemm_ffn2",
              7: "postchain", 8: "stack"}

EXPORTS = ("tfl_default_options", "tfl_workspace_bytes", "tfl_create", "tfl_forward", "tfl_forward_bf16",
           "tfl_forward_host", "tfl_forward_streamed",
           "tfl_attn_create", "tfl_attn_forward", "tfl_attn_backward", "tfl_attn_status", "tfl_attn_destroy",
           "tfl_status", "tfl_destroy", "tfl_last_error", "tfl_profile_forward", "tfl_launch_count",
           "tfl_probe_wait_timeout", "tfl_forward_noalloc", "tfl_selftest_gelu")

NOALLOC_SCRATCH_BYTES = 32 << 20


class TflShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("S", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("n_layers", ctypes.c_int32),
                ("norm_placement", ctypes.c_int32)]


_LW_FIELDS = ("wq", "bq", "wk", "bk", "wv", "bv", "wo", "bo", "ln1_g", "ln1_b", "ln2_g", "ln2_b",
              "w1", "b1", "w2", "b2")


class TflLayerWeights(ctypes.Structure):
    _fields_ = [(f, ctypes.c_void_p) for f in _LW_FIELDS]


class TflWeights(ctypes.Structure):
    _fields_ = [("layers", ctypes.POINTER(TflLayerWeights)), ("n_layers", ctypes.c_int32),
                ("lnf_g", ctypes.c_void_p), ("lnf_b", ctypes.c_void_p)]


class TflOptions(ctypes.Structure):
    _fields_ = [("precision", ctypes.c_int32), ("ln_eps", ctypes.c_float), ("wait_timeout_ns", ctypes.c_int64),
                ("max_workspace_bytes", ctypes.c_int64), ("use_graph", ctypes.c_int32),
                ("whole_stack", ctypes.c_int32), ("fp8_corrections", ctypes.c_int32)]


class TflError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"tfl error {code}: {msg}")
        self.code = code


_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the C-ABI library (once).  Raises ImportError if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"{p} not found: build it with `python -m attention_qkv_gemm_gb300.build` "
                          "(or __graft_entry__.build()); there is no non-CUDA fallback")
    lib = ctypes.CDLL(p)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.tfl_default_options.argtypes = [ctypes.POINTER(TflOptions)]
    lib.tfl_default_options.restype = ctypes.c_int
    lib.tfl_workspace_bytes.argtypes = [ctypes.POINTER(TflShape)]
    lib.tfl_workspace_bytes.restype = ctypes.c_size_t
    lib.tfl_create.argtypes = [ctypes.POINTER(TflShape), ctypes.POINTER(TflWeights), ctypes.POINTER(TflOptions),
                               ctypes.POINTER(vp)]
    lib.tfl_create.restype = ctypes.c_int
    lib.tfl_forward.argtypes = [vp, vp, vp, ctypes.c_int, vp, vp]
    lib.tfl_forward.restype = ctypes.c_int
    lib.tfl_forward_bf16.argtypes = [vp, vp, vp, ctypes.c_int, vp, vp]
    lib.tfl_forward_bf16.restype = ctypes.c_int
    lib.tfl_forward_noalloc.argtypes = [vp, vp, vp, ctypes.c_int, vp, vp]
    lib.tfl_forward_noalloc.restype = ctypes.c_int
    lib.tfl_forward_host.argtypes = [vp, vp, vp, ctypes.c_int, vp, vp]
    lib.tfl_forward_host.restype = ctypes.c_int
    lib.tfl_forward_streamed.argtypes = [vp, vp, vp, i64, ctypes.c_int, vp, vp]
    lib.tfl_forward_streamed.restype = ctypes.c_int
    lib.tfl_attn_create.argtypes = [i32, i32, i32, i32, ctypes.POINTER(vp)]
    lib.tfl_attn_create.restype = ctypes.c_int
    lib.tfl_attn_forward.argtypes = [vp, vp, vp, ctypes.c_int, vp, vp, vp]
    lib.tfl_attn_forward.restype = ctypes.c_int
    lib.tfl_attn_backward.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp]
    lib.tfl_attn_backward.restype = ctypes.c_int
    lib.tfl_attn_status.argtypes = [vp, vp]
    lib.tfl_attn_status.restype = ctypes.c_int
    lib.tfl_attn_destroy.argtypes = [vp]
    lib.tfl_attn_destroy.restype = None
    lib.tfl_status.argtypes = [vp, vp]
    lib.tfl_status.restype = ctypes.c_int
    lib.tfl_destroy.argtypes = [vp]
    lib.tfl_destroy.restype = None
    lib.tfl_last_error.argtypes = []
    lib.tfl_last_error.restype = ctypes.c_char_p
    lib.tfl_profile_forward.argtypes = [vp, vp, vp, ctypes.c_int, vp, vp, ctypes.POINTER(ctypes.c_float),
                                        ctypes.POINTER(i32), i32, ctypes.POINTER(i32)]
    lib.tfl_profile_forward.restype = ctypes.c_int
    lib.tfl_launch_count.argtypes = [vp, ctypes.c_int]
    lib.tfl_launch_count.restype = ctypes.c_int
    lib.tfl_selftest_gelu.argtypes = [i32, ctypes.POINTER(ctypes.c_float), vp]
    lib.tfl_selftest_gelu.restype = ctypes.c_int
    lib.tfl_probe_wait_timeout.argtypes = [i64, vp]
    lib.tfl_probe_wait_timeout.restype = ctypes.c_int
    _lib = lib
    return lib


def tfl_last_error() -> str:
    return load().tfl_last_error().decode()


def _check(rc: int) -> int:
    if rc != TFL_OK:
        raise TflError(rc, tfl_last_error())
    return rc


def tfl_default_options() -> TflOptions:
    o = TflOptions()
    _check(load().tfl_default_options(ctypes.byref(o)))
    return o


def tfl_workspace_bytes(shape: TflShape) -> int:
    return int(load().tfl_workspace_bytes(ctypes.byref(shape)))


def tfl_create(shape: TflShape, layer_ptrs: Sequence[dict], lnf_g: int, lnf_b: int,
               options: Optional[TflOptions] = None) -> int:
    """Create a handle.  ``layer_ptrs``: per layer a dict field -> pointer (int)."""
    arr = (TflLayerWeights * len(layer_ptrs))()
    for i, d in enumerate(layer_ptrs):
        for f in _LW_FIELDS:
            setattr(arr[i], f, d[f])
    w = TflWeights(arr, len(layer_ptrs), lnf_g, lnf_b)
    h = ctypes.c_void_p()
    _check(load().tfl_create(ctypes.byref(shape), ctypes.byref(w),
                             ctypes.byref(options) if options is not None else None, ctypes.byref(h)))
    return h.value


def tfl_forward(handle: int, x: int, lengths: Optional[int], causal: int, out: int, stream: int = 0) -> None:
    _check(load().tfl_forward(handle, x, lengths, int(causal), out, stream))


def tfl_forward_bf16(handle: int, x: int, lengths: Optional[int], causal: int, out: int, stream: int = 0) -> None:
    """The forward with bf16 model inputs and outputs (device pointers to bf16 [B, S, D])."""
    _check(load().tfl_forward_bf16(handle, x, lengths, int(causal), out, stream))


def tfl_forward_noalloc(handle: int, x: int, lengths: Optional[int], causal: int, out: int, stream: int = 0) -> None:
    """The forward with its intermediates in the library's fixed device array (no allocation)."""
    _check(load().tfl_forward_noalloc(handle, x, lengths, int(causal), out, stream))


def tfl_forward_host(handle: int, x: int, lengths: Optional[int], causal: int, out: int, stream: int = 0) -> int:
    """Returns the status code (0 or a device-side error), raising on call errors."""
    rc = load().tfl_forward_host(handle, x, lengths, int(causal), out, stream)
    if rc not in (TFL_OK, TFL_ERR_DEVICE_TIMEOUT, TFL_ERR_BAD_LENGTHS):
        raise TflError(rc, tfl_last_error())
    return rc


def tfl_forward_streamed(handle: int, x: int, lengths: Optional[int], n_seq: int, causal: int, out: int,
                         stream: int = 0) -> None:
    """n_seq sequences from pinned host x to pinned host out, streamed through the handle in
    slices of its batch size (asynchronous on ``stream``)."""
    _check(load().tfl_forward_streamed(handle, x, lengths, int(n_seq), int(causal), out, stream))


def tfl_attn_create(B: int, S: int, n_heads: int, head_dim: int) -> int:
    h = ctypes.c_void_p()
    _check(load().tfl_attn_create(int(B), int(S), int(n_heads), int(head_dim), ctypes.byref(h)))
    return h.value


def tfl_attn_forward(handle: int, qkv: int, lengths: Optional[int], causal: int, o: int, lse: int,
                     stream: int = 0) -> None:
    _check(load().tfl_attn_forward(handle, qkv, lengths, int(causal), o, lse, stream))


def tfl_attn_backward(handle: int, qkv: int, o: int, dout: int, lse: int, lengths: Optional[int], causal: int,
                      dqkv: int, stream: int = 0) -> None:
    _check(load().tfl_attn_backward(handle, qkv, o, dout, lse, lengths, int(causal), dqkv, stream))


def tfl_attn_status(handle: int, stream: int = 0) -> int:
    return load().tfl_attn_status(handle, stream)


def tfl_attn_destroy(handle: int) -> None:
    if handle:
        load().tfl_attn_destroy(handle)


def tfl_status(handle: int, stream: int = 0) -> int:
    return load().tfl_status(handle, stream)


def tfl_destroy(handle: int) -> None:
    if handle:
        load().tfl_destroy(handle)


def tfl_launch_count(handle: int, causal: int) -> int:
    return int(load().tfl_launch_count(handle, int(causal)))


def tfl_profile_forward(handle: int, x: int, lengths: Optional[int], causal: int, out: int, stream: int = 0,
                        cap: int = 512):
    """Eager forward with an event around each launch: list of (kind_name, ms)."""
    ms = (ctypes.c_float * cap)()
    kinds = (ctypes.c_int32 * cap)()
    n = ctypes.c_int32()
    _check(load().tfl_profile_forward(handle, x, lengths, int(causal), out, stream, ms, kinds, cap, ctypes.byref(n)))
    return [(KIND_NAMES.get(kinds[i], str(kinds[i])), float(ms[i])) for i in range(min(n.value, cap))]


def tfl_selftest_gelu(n: int = 1 << 20, stream: int = 0) -> float:
    """Largest |GELU(A&S 7.1.26) - GELU(erff)| on the GPU over n points of [-12, 12]."""
    v = ctypes.c_float()
    _check(load().tfl_selftest_gelu(int(n), ctypes.byref(v), stream))
    return float(v.value)


def tfl_probe_wait_timeout(timeout_ns: int, stream: int = 0) -> int:
    return int(load().tfl_probe_wait_timeout(int(timeout_ns), stream))


# ----------------------------------------------------------------------------
# Convenience wrapper over torch device tensors
# ----------------------------------------------------------------------------

class TransformerStack:
    """Owns a handle built from float32 parameters (numpy arrays or tensors).

    ``params`` has ``layers`` (objects with the 16 fields of
    ``tfl_layer_weights``) and ``lnf_g`` / ``lnf_b``; values are copied once
    by ``tfl_create`` and may be freed afterwards.
    """

    def __init__(self, B: int, S: int, d_model: int, n_heads: int, d_ff: int, n_layers: int, params,
                 norm_placement: int = 0, options: Optional[TflOptions] = None):
        import numpy as np
        self.shape = TflShape(B, S, d_model, n_heads, d_ff, n_layers, norm_placement)
        keep = []

        def ptr(a):
            if hasattr(a, "data_ptr"):
                t = a.detach().float().contiguous()
                keep.append(t)
                return t.data_ptr()
            arr = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
            keep.append(arr)
            return arr.ctypes.data

        layer_ptrs = [{f: ptr(getattr(L, f)) for f in _LW_FIELDS} for L in params.layers]
        self.handle = tfl_create(self.shape, layer_ptrs, ptr(params.lnf_g), ptr(params.lnf_b), options)
        del keep

    def forward(self, x, lengths=None, causal: bool = True, out=None, stream: Optional[int] = None):
        """x: torch float32 or bfloat16 CUDA [B, S, D]; lengths: int32 CUDA [B] or None.
        Returns out, in x's dtype."""
        import torch
        if out is None:
            out = torch.empty_like(x)
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        fn = tfl_forward_bf16 if x.dtype == torch.bfloat16 else tfl_forward
        if out.dtype != x.dtype:
            raise ValueError("out must have x's dtype")
        fn(self.handle, x.data_ptr(), None if lengths is None else lengths.data_ptr(), int(causal), out.data_ptr(),
           stream)
        return out

    def status(self, stream: Optional[int] = None) -> int:
        import torch
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        return tfl_status(self.handle, stream)

    def close(self):
        if getattr(self, "handle", None):
            tfl_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
