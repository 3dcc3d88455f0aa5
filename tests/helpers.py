"""Shared helpers for the GPU parity tests: build inputs, run the C-ABI path."""
from __future__ import annotations

import numpy as np

import oracle
import synth


def run_gpu(shape: synth.Shape, prm, x: np.ndarray, lens, causal: bool, norm_placement: int = 0,
            use_graph: bool = True, repeat: int = 1, fp8_corrections: int = None):
    """Run the library forward on cuda:0; returns (out numpy, status code)."""
    import torch
    import attention_qkv_gemm_gb300 as pkg

    opts = pkg.tfl_default_options()
    opts.use_graph = 1 if use_graph else 0
    if fp8_corrections is not None:
        opts.fp8_corrections = fp8_corrections
    m = pkg.TransformerStack(shape.B, shape.S, shape.d_model, shape.n_heads, shape.d_ff, shape.n_layers, prm,
                             norm_placement=norm_placement, options=opts)
    try:
        xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
        ld = None if lens is None else torch.from_numpy(np.asarray(lens, dtype=np.int32)).cuda()
        out = torch.full_like(xd, float("nan"))
        for _ in range(repeat):
            m.forward(xd, ld, causal=causal, out=out)
        rc = m.status()
        return out.cpu().numpy(), rc
    finally:
        m.close()


def gate_report(u: np.ndarray, r: np.ndarray) -> str:
    ok = oracle.gate(u, r)
    d = np.abs(u - r)
    return (f"fail {int((~ok).sum())}/{ok.size}, max|d| {d.max():.3e}, "
            f"first bad {np.argwhere(~ok)[:3].tolist()}")


def assert_gate(u: np.ndarray, r: np.ndarray, what: str = ""):
    ok = oracle.gate(u, r)
    assert np.isfinite(u).all(), f"{what}: non-finite output"
    assert ok.all(), f"{what}: {gate_report(u, r)}"
