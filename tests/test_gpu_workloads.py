"""GPU parity at the five benchmark shapes, element by element, over 25 seeds.

"Transformerkernel" (Challenges) ran its checks over 25 trials and warns that the
worst element of a run grows like sigma * sqrt(2 ln N) with the number N of
elements checked, so a gate that samples a few sequences understates the error
the rule has to absorb.  The GPU runs the whole batch at full size through the
C ABI, in the launch configuration the benchmark times (graph replay), and the
fp64 oracle then checks it with the graded rule |u-r| <= 2e-3 or <= 0.02|r|:
  * B=1 S=128, B=64 S=1024 and B=16 S=512: every element of every sequence,
    seeds 0..24;
  * B=10000 S=128: every element of every sequence for seeds 0..4, and for
    seeds 5..24 whole sampled sequences (always the longest and the shortest),
    with every padded row of the whole batch checked to be exactly zero;
  * B=32 S=100000 (one causal layer): 2 sequences x 64 query rows per seed,
    always including rows 0 and S-1 (exact: with one causal layer a row depends
    only on the keys before it); seeds 0..4 by default (about 20 s each), more
    with --s100k-seeds N.
Seeds drive both weights and inputs.  The worst ratio |u-r| / max(2e-3,
0.02|r|) over all seeds is printed for the record.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import gate_report

pytestmark = pytest.mark.gpu

SEEDS = list(range(25))
FULL_SEEDS_B10000 = 5


def _run_full(shape, prm, x, lens):
    import torch
    import attention_qkv_gemm_gb300 as pkg
    m = pkg.TransformerStack(shape.B, shape.S, shape.d_model, shape.n_heads, shape.d_ff, shape.n_layers, prm)
    try:
        xd = torch.from_numpy(x).cuda()
        ld = torch.from_numpy(lens).cuda()
        out = m.forward(xd, ld, causal=shape.causal)
        rc = m.status()
        assert rc == 0, pkg.tfl_last_error()
        return out
    finally:
        m.close()


def _ratio(u, r):
    return float(np.max(np.abs(u - r) / np.maximum(2e-3, 0.02 * np.abs(r))))


def _oracle_all(shape, prm, x, lens):
    """fp64 oracle output of every sequence of the batch."""
    if shape.d_model <= 128:
        # many small array operations: worker processes, one sequence group per task
        chunk = 1 if shape.S >= 512 else 128
        return oracle.forward_batched(prm, shape.n_heads, x, lens, shape.causal, chunk=chunk, processes=True)
    # large projections: one batch, multi-threaded BLAS in this process
    return oracle.forward_batched(prm, shape.n_heads, x, lens, shape.causal, chunk=shape.B)


def _padded_rows_zero(out, lens, S, seed):
    import torch
    pad = np.arange(S)[None, :] >= lens[:, None]
    if pad.any():
        padmask = torch.from_numpy(pad).cuda()
        assert bool((out[padmask] == 0).all()), f"seed {seed}: padded rows not zero"


def _check_every_element(wl_index, seeds):
    shape = synth.WORKLOADS[wl_index]
    worst = 0.0
    for seed in seeds:
        prm = synth.params(seed, shape)
        lens = synth.lengths(seed, shape)
        x = synth.input_x(seed, shape)
        out = _run_full(shape, prm, x, lens)
        _padded_rows_zero(out, lens, shape.S, seed)
        u = out.cpu().numpy()
        del out
        r = _oracle_all(shape, prm, x, lens)
        assert np.isfinite(u).all(), f"{shape.name} seed {seed}: non-finite output"
        ok = oracle.gate(u, r)
        assert ok.all(), f"{shape.name} seed {seed}: {gate_report(u, r)}"
        worst = max(worst, _ratio(u, r))
    print(f"\n{shape.name}: worst |u-r|/budget over {len(seeds)} seeds, every element = {worst:.3f}")
    return worst


def _check_sequences(wl_index, n_seq, seeds):
    shape = synth.WORKLOADS[wl_index]
    worst = 0.0
    for seed in seeds:
        prm = synth.params(seed, shape)
        lens = synth.lengths(seed, shape)
        x = synth.input_x(seed, shape)
        out = _run_full(shape, prm, x, lens)
        _padded_rows_zero(out, lens, shape.S, seed)
        rng = np.random.default_rng(1000 + seed)
        pick = {int(np.argmax(lens)), int(np.argmin(lens))}
        while len(pick) < min(n_seq, shape.B):
            pick.add(int(rng.integers(shape.B)))
        bsel = np.array(sorted(pick))
        u = out[bsel].cpu().numpy()
        del out
        r = oracle.forward_batched(prm, shape.n_heads, x[bsel], lens[bsel], shape.causal)
        assert np.isfinite(u).all()
        assert oracle.gate(u, r).all(), f"{shape.name} seed {seed} sequences {bsel.tolist()}: {gate_report(u, r)}"
        worst = max(worst, _ratio(u, r))
    print(f"\n{shape.name}: worst |u-r|/budget over {len(seeds)} seeds ({n_seq} sampled sequences) = {worst:.3f}")


def test_workload_b1_s128_all_elements():
    _check_every_element(0, SEEDS)


def test_workload_b64_s1024_ragged_all_elements():
    _check_every_element(1, SEEDS)


def test_workload_b10000_s128_keymask_all_elements():
    _check_every_element(2, list(range(FULL_SEEDS_B10000)))


def test_workload_b10000_s128_keymask_sampled_sequences():
    _check_sequences(2, 16, list(range(FULL_SEEDS_B10000, 25)))


def test_workload_b16_s512_d1024_all_elements():
    _check_every_element(3, SEEDS)


def test_workload_b32_s100000_sampled_rows(request):
    import torch
    import attention_qkv_gemm_gb300 as pkg
    shape = synth.WORKLOADS[4]
    n_seeds = request.config.getoption("--s100k-seeds")
    worst = 0.0
    for seed in range(n_seeds):
        prm = synth.params(seed, shape)
        lens = synth.lengths(seed, shape)
        x = synth.input_x(seed, shape)
        m = pkg.TransformerStack(shape.B, shape.S, shape.d_model, shape.n_heads, shape.d_ff, shape.n_layers, prm)
        try:
            xd = torch.from_numpy(x).cuda()
            ld = torch.from_numpy(lens).cuda()
            out = m.forward(xd, ld, causal=True)
            assert m.status() == 0, pkg.tfl_last_error()
            rng = np.random.default_rng(2000 + seed)
            bsel = np.sort(rng.choice(shape.B, 2, replace=False))
            rows = np.unique(np.concatenate([[0, shape.S - 1], rng.choice(shape.S, 62, replace=False)]))
            u = out[torch.from_numpy(bsel).cuda()][:, torch.from_numpy(rows).cuda()].cpu().numpy()
        finally:
            m.close()
            del xd
        r = oracle.forward(prm, shape.n_heads, x[bsel], lens[bsel], True, rows=rows)
        assert oracle.gate(u, r).all(), f"seed {seed}: {gate_report(u, r)}"
        worst = max(worst, _ratio(u, r))
    print(f"\n{shape.name}: worst |u-r|/budget over {n_seeds} seeds (sampled rows) = {worst:.3f}")
