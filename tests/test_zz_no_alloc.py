"""tfl_forward_noalloc: the forward for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc when they run the forward -- for example
code running inside another component's CUDA-graph capture, or under a host
framework whose pool owns the device memory.  tfl_forward_noalloc keeps every
intermediate of the forward in one fixed device array inside the library
instead of the handle's workspace.  It runs the same kernels on the same
inputs as tfl_forward, and the forward is deterministic, so these tests ask
for bit equality with tfl_forward (same handle, same inputs), on two calls in
a row with different inputs and lengths, with a call from another handle of
another shape and precision in between (the array is shared by every handle
on the device and keeps the last call's contents).  Both launch sequences are
covered: the fused chain (d_model 128) and the separate GEMM + row-kernel
sequence (d_model 256).  This file is collected last on purpose.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def _stack(shape, seed, precision=2):
    import attention_qkv_gemm_gb300 as pkg
    opts = pkg.tfl_default_options()
    opts.precision = precision
    prm = synth.params(seed, shape, ln_affine="random")
    return pkg.TransformerStack(shape.B, shape.S, shape.d_model, shape.n_heads, shape.d_ff, shape.n_layers, prm,
                                options=opts)


def _noalloc(m, x, lens, causal):
    import torch
    import attention_qkv_gemm_gb300 as pkg
    out = torch.full_like(x, float("nan"))
    pkg.tfl_forward_noalloc(m.handle, x.data_ptr(), None if lens is None else lens.data_ptr(), int(causal),
                            out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert m.status() == 0, pkg.tfl_last_error()
    return out


@pytest.mark.parametrize("D,H,F", [(128, 4, 512), (256, 4, 512)])
def test_noalloc_bit_equal_to_tfl_forward_across_handles(D, H, F):
    import torch
    shape = synth.Shape(2, 200, D, H, F, 2, True)
    other = synth.Shape(3, 328, 128, 4, 384, 1, False)  # another layout in the shared array
    m = _stack(shape, 7)
    m2 = _stack(other, 8, precision=1)
    try:
        cases = [(synth.input_x(7, shape), np.array([200, 61], dtype=np.int32)),
                 (synth.input_x(8, shape), np.array([129, 200], dtype=np.int32))]
        for i, (x_np, lens_np) in enumerate(cases):
            x = torch.from_numpy(x_np).cuda()
            lens = torch.from_numpy(lens_np).cuda()
            ref = m.forward(x, lens, causal=True)
            out = _noalloc(m, x, lens, True)
            u, r = out.cpu().numpy(), ref.cpu().numpy()
            assert np.isfinite(u).all()
            np.testing.assert_array_equal(u, r)
            for b in range(shape.B):
                assert np.all(u[b, lens_np[b]:] == 0.0)
            if i == 0:
                # the other handle leaves its own contents in the array
                x2 = torch.from_numpy(synth.input_x(9, other) * np.float32(50.0)).cuda()
                l2 = torch.tensor([328, 5, 200], dtype=torch.int32, device="cuda")
                o2 = _noalloc(m2, x2, l2, False)
                np.testing.assert_array_equal(o2.cpu().numpy(), m2.forward(x2, l2, causal=False).cpu().numpy())
    finally:
        m.close()
        m2.close()


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import torch
    import attention_qkv_gemm_gb300 as pkg
    shape = synth.Shape(16, 1024, 128, 4, 512, 1, True)  # ~64 MiB of intermediates
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
