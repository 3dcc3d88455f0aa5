"""tfl_forward_streamed: a batch in pinned host memory, streamed through the device in slices.

"Shape-specialized Transformer Inference on Commodity GPUs" (How we built it)
runs its S = 100000 case with the input in host RAM, batch slices streamed
through the device and the outputs streamed back.  Here the slices run through a
handle whose batch size is the slice size, with copies overlapping compute.
  * The slicing must not change the arithmetic: at d_model 1024 every kernel's
    result for a row is independent of the row's place in the batch, so the
    streamed output equals tfl_forward over the whole batch bit for bit, with a
    partial last slice and ragged lengths.
  * d_model 128, lengths mixed: every element against the fp64 oracle.
  * The B=32 S=100000 workload streamed in slices of 4 sequences: 2 sequences x
    64 query rows against the oracle (exact: one causal layer).
"""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import assert_gate

pytestmark = pytest.mark.gpu


def _pinned(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def _streamed(shape, prm, slice_b, x, lens, causal):
    """Run n = x.shape[0] sequences through a handle of batch size slice_b."""
    import torch
    import attention_qkv_gemm_gb300 as pkg
    m = pkg.TransformerStack(slice_b, shape.S, shape.d_model, shape.n_heads, shape.d_ff, shape.n_layers, prm)
    try:
        hx = _pinned(x)
        ho = torch.full_like(hx, float("nan")).pin_memory()
        st = torch.cuda.current_stream().cuda_stream
        pkg.tfl_forward_streamed(m.handle, hx.data_ptr(), None if lens is None else _pinned(lens).data_ptr(),
                                 x.shape[0], int(causal), ho.data_ptr(), st)
        assert m.status() == 0, pkg.tfl_last_error()
        return ho.numpy().copy()
    finally:
        m.close()


def test_streamed_equals_whole_batch_forward_bitwise():
    import torch
    import attention_qkv_gemm_gb300 as pkg
    shape = synth.Shape(5, 700, 1024, 16, 1024, 2, True)
    prm = synth.params(21, shape, ln_affine="random")
    x = synth.input_x(21, shape)
    lens = np.array([700, 3, 511, 0, 640], dtype=np.int32)
    u = _streamed(shape, prm, 2, x, lens, True)          # slices of 2, 2, 1
    m = pkg.TransformerStack(shape.B, shape.S, shape.d_model, shape.n_heads, shape.d_ff, shape.n_layers, prm)
    try:
        ref = m.forward(torch.from_numpy(x).cuda(), torch.from_numpy(lens).cuda(), causal=True)
        assert m.status() == 0
        ref = ref.cpu().numpy()
    finally:
        m.close()
    np.testing.assert_array_equal(u, ref)
    assert np.all(u[3] == 0.0)


def test_streamed_d128_against_oracle():
    shape = synth.Shape(7, 300, 128, 4, 512, 2, False)
    prm = synth.params(22, shape, ln_affine="random")
    x = synth.input_x(22, shape)
    lens = np.array([300, 17, 129, 256, 1, 300, 200], dtype=np.int32)
    u = _streamed(shape, prm, 3, x, lens, False)          # slices of 3, 3, 1
    r = oracle.forward_batched(prm, shape.n_heads, x, lens, False)
    for b in range(shape.B):
        assert np.all(u[b, lens[b]:] == 0.0)
    assert_gate(u, r, "streamed B7 S300 D128 key mask")


def test_streamed_b32_s100000_sampled_rows():
    shape = synth.WORKLOADS[4]
    seed = 0
    prm = synth.params(seed, shape)
    x = synth.input_x(seed, shape)
    u = _streamed(shape, prm, 4, x, None, True)
    rng = np.random.default_rng(3000 + seed)
    bsel = np.sort(rng.choice(shape.B, 2, replace=False))
    rows = np.unique(np.concatenate([[0, shape.S - 1], rng.choice(shape.S, 62, replace=False)]))
    r = oracle.forward(prm, shape.n_heads, x[bsel], None, True, rows=rows)
    assert_gate(u[bsel][:, rows], r, "streamed B32 S100000")
