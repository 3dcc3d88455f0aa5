"""bench.py's accounting, checked against closed forms (CPU).

Algorithmic FLOPs per forward count only the work the method must do: the four
projections on valid rows (2 * rows * (3D*D + D*D + 2*D*F) per layer) and, for
attention, 4 * head_dim FLOPs (QK^T and P V) per allowed (query, key) pair and
head.  With full lengths and a causal mask a sequence of S tokens has
S (S + 1) / 2 allowed pairs.
"""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def _full(shape):
    return np.full(shape.B, shape.S, dtype=np.int32)


@pytest.mark.parametrize("idx", [0, 3, 4])
def test_algorithmic_flops_full_lengths_closed_form(idx):
    shape = synth.WORKLOADS[idx]
    B, S, D, H, F, L = shape.B, shape.S, shape.d_model, shape.n_heads, shape.d_ff, shape.n_layers
    a = bench.algorithmic(shape, _full(shape), True)
    lin = 2.0 * B * S * (4 * D * D + 2 * D * F) * L
    att = 4.0 * (D // H) * H * B * S * (S + 1) / 2 * L
    assert a["valid_tokens"] == B * S
    assert a["linear_flops"] == pytest.approx(lin, rel=1e-12)
    assert a["attn_flops"] == pytest.approx(att, rel=1e-12)
    assert a["attn_exps_per_launch"] == pytest.approx(H * B * S * (S + 1) / 2, rel=1e-12)


def test_algorithmic_flops_match_the_workload_table():
    # totals per forward, GFLOP: B16 S512 D1024 ~ 859, B32 S100000 D1024 ~ 735 900, B1 S128 ~ 0.218
    got = {i: (lambda s: sum(bench.algorithmic(s, _full(s), True)[k] for k in ("linear_flops", "attn_flops")))(
        synth.WORKLOADS[i]) / 1e9 for i in (0, 3, 4)}
    assert got[0] == pytest.approx(0.218, rel=0.01)
    assert got[3] == pytest.approx(859.1, rel=0.001)
    assert got[4] == pytest.approx(735_900, rel=0.001)


def test_key_padding_counts_only_valid_pairs():
    shape = synth.Shape(2, 128, 128, 4, 512, 1, False, 32, 128)
    lens = np.array([100, 7], dtype=np.int32)
    a = bench.algorithmic(shape, lens, False)
    assert a["valid_tokens"] == 107
    assert a["pairs"] == 100 * 100 + 7 * 7


def test_gemm_flops_per_launch():
    shape = synth.WORKLOADS[3]
    assert bench.gemm_flops("gemm_ffn2", shape, 8192) == 2.0 * 8192 * 1024 * 4096
    assert bench.gemm_flops("gemm_qkv", shape, 8192) == 2.0 * 8192 * 3072 * 1024
    assert bench.gemm_flops("attention", shape, 8192) is None


def test_chain_bytes_per_valid_token():
    # fused chain at d_model 128, averaged over a forward's four launches:
    # (3 x (256 + 512 + 512 + 768) + (256 + 512 + 512)) / 4 = 1856 bytes per valid token
    shape = synth.WORKLOADS[1]
    assert bench.kernel_bytes("postchain", shape, 1.0) == pytest.approx(1856.0)


def test_custom_shape_and_row_sample():
    s = bench.custom_shape("2,16384,1024,16,4096,1,1")
    assert (s.B, s.S, s.d_model, s.n_heads, s.d_ff, s.n_layers, s.causal) == (2, 16384, 1024, 16, 4096, 1, True)
    s2 = bench.custom_shape("4,200,128,4,512,2,0,32,200")
    assert (s2.causal, s2.len_lo, s2.len_hi) == (False, 32, 200)
    with pytest.raises(SystemExit):
        bench.custom_shape("1,2,3")
    rows = bench.oracle_rows(synth.WORKLOADS[4])
    assert rows is not None and len(rows) == bench.ORACLE_ROWS
    assert rows[0] == 0 and rows[-1] == synth.WORKLOADS[4].S - 1 and np.all(np.diff(rows) > 0)
    assert bench.oracle_rows(synth.WORKLOADS[1]) is None  # short sequences: whole sequences


def test_live_tiles_and_chain_executed_mmas():
    # B2 S256, lengths 256 and 1: tiles 0-1 hold sequence 0; tile 2 holds sequence 1's only
    # valid row (and its key rows up to 64); tile 3 is all padding
    shape = synth.Shape(2, 256, 128, 4, 512, 3, True)
    lens = np.array([256, 1], dtype=np.int32)
    assert bench.live_tiles(shape, lens) == 3
    # per live tile: o_proj 16 + FFN 48 per 128-wide chunk in every launch, QKV 72 in all but the last
    per_tile = 3 * (16 + 48 * 4) + 2 * 72
    assert bench.chain_executed_flops(shape, lens) == pytest.approx(3 * per_tile * 2.0 * 128 * 128 * 16)


def test_whole_stack_accounting():
    shape = synth.Shape(3, 128, 128, 4, 384, 2, False)
    lens = np.array([128, 0, 5], dtype=np.int32)
    # two non-empty sequences x two layers x (QKV 72 + 4 heads x 5 + o_proj 16 + 48 per chunk)
    per_layer = 72 + 20 + 16 + 48 * 3
    assert bench.stack_executed_flops(shape, lens) == pytest.approx(2 * 2 * per_layer * 2.0 * 128 * 128 * 16)
    valid = float(lens.sum())
    weights = 2 * (4 * 128 * 128 + 2 * 128 * 384) * 2 * 2
    assert bench.stack_bytes(shape, valid) == pytest.approx(valid * 512 + 3 * 128 * 512 + weights)
    assert bench.forward_bytes(shape, valid) == pytest.approx(bench.stack_bytes(shape, valid))


def test_e2e_slice_rule():
    big, small, many = synth.WORKLOADS[4], synth.WORKLOADS[1], synth.WORKLOADS[2]
    assert bench.e2e_slice(big, 0) == 1          # 13 GB of input: a thirty-second of the batch
    assert bench.e2e_slice(small, 0) == 0        # 33.5 MB: no slicing
    assert bench.e2e_slice(many, 0) == 0         # B10000 S128, 655 MB: no slicing
    assert bench.e2e_slice(big, -1) == 0 and bench.e2e_slice(big, 5) == 5
    assert bench.e2e_slice(small, 100) == small.B


def test_compute_dtype_names_the_fp8_correction_products():
    assert bench.compute_dtype(synth.WORKLOADS[4]) == "f16+e4m3"
    assert bench.compute_dtype(synth.WORKLOADS[3]) == "f16+e4m3"
    assert bench.compute_dtype(synth.WORKLOADS[1]) == "f16"


def test_attention_cycles_copy_applies_and_builds(tmp_path):
    # --attn-cycles instruments attention.cu by inserting counters at fixed anchors; every
    # anchor must still match the kernel exactly once, and the copy must compile with the same
    # launch-register count as the library (its setmaxnreg split needs it)
    import subprocess
    from attention_qkv_gemm_gb300 import build as libbuild
    with open(f"{libbuild.CSRC}/attention.cu") as f:
        src = f.read()
    out = bench.attention_cycles_source(src)
    assert out.count("atomicAdd(&g_attn_cycles[") == 9
    assert 'extern "C" int tfl_attn_cycles_fetch' in out
    cu = tmp_path / "attention_cycles.cu"
    cu.write_text(out)
    r = subprocess.run([libbuild._nvcc(), *libbuild.ARCH, *libbuild.FLAGS, "-Xptxas", "-v", "-c", str(cu),
                        "-o", str(tmp_path / "a.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    libbuild.check_launch_registers(r.stdout + r.stderr)


def test_attention_cycles_copy_refuses_a_changed_kernel():
    with pytest.raises(RuntimeError, match="anchor"):
        bench.attention_cycles_source("namespace tfl {\n}  // namespace tfl\n")


def test_attention_cycles_report_divides_per_subblock_and_warp():
    # two CTAs of 10 sub-blocks: issuer counters summed over the CTAs, softmax counters over the
    # four warps of each CTA as well
    c = [0.0] * 16
    c[4] = c[12] = 20.0
    c[0], c[1], c[2], c[3] = 1000 * 20.0, 300 * 20.0, 50 * 20.0, 600 * 20.0
    c[8], c[9], c[10], c[11] = 900 * 20.0, 200 * 20.0, 80 * 20.0, 500 * 20.0
    c[5], c[6], c[7], c[13] = (v * 20 * 4 for v in (1000.0, 150.0, 980.0, 15.0))
    r = bench.attention_cycles_report(c, 2, 16384, 16, 64, 1, 3)
    assert r["pv_thread"] == {"total": 1000.0, "waiting_for_p": 300.0, "waiting_for_kv": 50.0, "issuing": 600.0}
    assert r["qk_thread"] == {"total": 900.0, "waiting_for_pv": 200.0, "waiting_for_kv": 80.0, "issuing": 500.0}
    assert r["softmax_warp"] == {"total": 1000.0, "waiting_for_s": 150.0, "subblock_loop": 980.0, "output": 15.0}
    assert r["config"]["launches"] == 3
