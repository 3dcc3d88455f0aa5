"""The seeded input generator: determinism, slicing, distributions (CPU)."""
import json
import os

import numpy as np

import synth

HERE = os.path.dirname(__file__)


def test_workload_table_matches_golden():
    g = json.load(open(os.path.join(HERE, "golden", "workloads.json")))
    assert len(g["workloads"]) == len(synth.WORKLOADS)
    for w, s in zip(g["workloads"], synth.WORKLOADS):
        assert (w["B"], w["S"], w["d_model"], w["n_heads"], w["d_ff"], w["n_layers"], w["causal"]) == \
            (s.B, s.S, s.d_model, s.n_heads, s.d_ff, s.n_layers, s.causal)
        assert (w["len"] is None) == (s.len_lo is None)
        if w["len"] is not None:
            assert w["len"] == [s.len_lo, s.len_hi]


def test_normal_is_deterministic_and_slice_consistent():
    a = synth.normal(3, "x", 10000)
    b = synth.normal(3, "x", 10000)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(synth.normal(3, "x", 100, start=5000), a[5000:5100])
    assert not np.array_equal(a, synth.normal(4, "x", 10000))
    assert not np.array_equal(a, synth.normal(3, "y", 10000))
    big = synth.normal(7, "z", (1 << 22) + 123, threads=3)
    np.testing.assert_array_equal(big[(1 << 22):], synth.normal(7, "z", 123, start=1 << 22))


def test_normal_moments():
    z = synth.normal(1, "m", 1 << 20).astype(np.float64)
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1) < 5e-3
    assert abs(np.mean(z ** 4) - 3) < 0.05


def test_lengths_and_batch_slices():
    s = synth.WORKLOADS[1]
    L = synth.lengths(0, s)
    assert L.dtype == np.int32 and L.min() >= 512 and L.max() <= 1024
    assert len(np.unique(L)) > 20
    assert np.all(synth.lengths(0, synth.WORKLOADS[0]) == 128)
    small = synth.Shape(4, 16, 32, 2, 64, 1, True)
    x = synth.input_x(2, small)
    np.testing.assert_array_equal(synth.input_x(2, small, batches=np.array([2, 0])), x[[2, 0]])


def test_param_scales():
    s = synth.Shape(1, 8, 256, 4, 1024, 1, True)
    p = synth.params(0, s).layers[0]
    assert abs(p.wq.std() - 1 / 16) < 2e-3 and abs(p.w2.std() - 1 / 32) < 1e-3
    assert abs(p.b1.std() - 0.02) < 3e-3
    assert np.all(p.ln1_g == 1) and np.all(p.ln2_b == 0)
