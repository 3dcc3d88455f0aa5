"""The MUFU exponential rate that bench.py takes as the attention kernel's peak.

bench.py holds head_dim-32 attention against 32 ex2.approx.f32 results per clock
per SM (times the SM count and the maximum SM clock).  This test builds the
throughput probe tests/probes/ex2_rate.cu with nvcc, runs it on the GPU and
checks the measured rate is that figure (within 10 %).
"""
import os
import re
import shutil
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_ex2_rate_matches_the_bench_peak():
    import bench
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "ex2_rate")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe,
                        os.path.join(HERE, "probes", "ex2_rate.cu")], check=True, capture_output=True, timeout=300)
        out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=120).stdout
    print("\n" + out)
    rates = [float(v) for v in re.findall(r"ex2\.approx\.f32 \(results\)\s+\d+ warps/SM:\s+([\d.]+)", out)]
    assert len(rates) == 2
    for r in rates:
        assert abs(r - bench.MUFU_PER_CLK_PER_SM) <= 0.1 * bench.MUFU_PER_CLK_PER_SM, out
