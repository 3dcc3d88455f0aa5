"""tfl_forward_noalloc: the forward for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc when they run the forward -- for example
code running inside another component's CUDA-graph capture, or under a host
framework whose pool owns the device memory.  tfl_forward_noalloc keeps every
intermediate of the forward in one fixed device array inside the library
instead of the handle's workspace.  These tests call it through the C ABI
and compare it with tfl_forward (same handle, same inputs) under the graded
rule used by every parity test here, on two calls in a row with different
inputs and lengths, so that contents left in the shared array by the first
call cannot leak into the second.  This file is collected last on purpose.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import gate_report

pytestmark = pytest.mark.gpu


def test_noalloc_matches_tfl_forward_on_two_calls_in_a_row():
    import torch
    import attention_qkv_gemm_gb300 as pkg
    shape = synth.Shape(2, 200, 128, 4, 512, 2, True)
    prm = synth.params(7, shape, ln_affine="random")
    m = pkg.TransformerStack(shape.B, shape.S, shape.d_model, shape.n_heads, shape.d_ff, shape.n_layers, prm)
    try:
        stream = torch.cuda.current_stream().cuda_stream
        cases = [(synth.input_x(7, shape), np.array([200, 61], dtype=np.int32)),
                 (synth.input_x(8, shape), np.array([129, 200], dtype=np.int32))]
        for x_np, lens_np in cases:
            x = torch.from_numpy(x_np).cuda()
            lens = torch.from_numpy(lens_np).cuda()
            ref = m.forward(x, lens, causal=True)
            out = torch.full_like(x, float("nan"))
            pkg.tfl_forward_noalloc(m.handle, x.data_ptr(), lens.data_ptr(), 1, out.data_ptr(), stream)
            assert m.status() == 0, pkg.tfl_last_error()
            u, r = out.cpu().numpy(), ref.cpu().numpy()
            assert np.isfinite(u).all()
            assert oracle.gate(u, r).all(), gate_report(u, r)
            for b in range(shape.B):
                assert np.all(u[b, lens_np[b]:] == 0.0)
    finally:
        m.close()


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import torch
    import attention_qkv_gemm_gb300 as pkg
    shape = synth.Shape(16, 1024, 128, 4, 512, 1, True)  # ~70 MiB of intermediates
    prm = synth.params(9, shape)
    assert pkg.tfl_workspace_bytes(pkg.TflShape(16, 1024, 128, 4, 512, 1, 0)) > pkg.NOALLOC_SCRATCH_BYTES
    m = pkg.TransformerStack(shape.B, shape.S, shape.d_model, shape.n_heads, shape.d_ff, shape.n_layers, prm)
    try:
        x = torch.zeros(shape.B, shape.S, shape.d_model, device="cuda")
        out = torch.empty_like(x)
        with pytest.raises(pkg.TflError) as ei:
            pkg.tfl_forward_noalloc(m.handle, x.data_ptr(), None, 1, out.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)
        assert ei.value.code == pkg.TFL_ERR_UNSUPPORTED
        assert "bytes of scratch" in str(ei.value)
    finally:
        m.close()
