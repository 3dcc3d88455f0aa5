"""The build's check on the attention kernels' launch register count (CPU).

attn_kernel<32> and attn_kernel<64> move registers between their two warpgroups with
setmaxnreg (64 and 192 a thread); that balances only at exactly 128 registers a thread at
launch, so the build refuses any other count rather than leave setmaxnreg.inc waiting on the
GPU.  These tests feed the check ptxas-style logs and check the library built here.
"""
import pytest

from attention_qkv_gemm_gb300 import build as b

LOG = """ptxas info    : Compiling entry function '_ZN3tfl11attn_kernelILi256EEEv14CUtensorMap_stS1_NS_8AttnArgsE' for 'sm_103a'
ptxas info    : Function properties for _ZN3tfl11attn_kernelILi256EEEv14CUtensorMap_stS1_NS_8AttnArgsE
    0 bytes stack frame, 0 bytes spill stores, 0 bytes spill loads
ptxas info    : Used 200 registers, used 1 barriers
ptxas info    : Compiling entry function '_ZN3tfl11attn_kernelILi64EEEv14CUtensorMap_stS1_NS_8AttnArgsE' for 'sm_103a'
ptxas info    : Function properties for _ZN3tfl11attn_kernelILi64EEEv14CUtensorMap_stS1_NS_8AttnArgsE
    0 bytes stack frame, 0 bytes spill stores, 0 bytes spill loads
ptxas info    : Used {r64} registers, used 1 barriers
ptxas info    : Compiling entry function '_ZN3tfl11attn_kernelILi32EEEv14CUtensorMap_stS1_NS_8AttnArgsE' for 'sm_103a'
ptxas info    : Function properties for _ZN3tfl11attn_kernelILi32EEEv14CUtensorMap_stS1_NS_8AttnArgsE
    0 bytes stack frame, 0 bytes spill stores, 0 bytes spill loads
ptxas info    : Used {r32} registers, used 1 barriers
"""


def test_launch_registers_parses_each_entry_function():
    regs = b.launch_registers(LOG.format(r64=128, r32=120))
    assert regs["_ZN3tfl11attn_kernelILi256EEEv14CUtensorMap_stS1_NS_8AttnArgsE"] == 200
    assert regs["_ZN3tfl11attn_kernelILi64EEEv14CUtensorMap_stS1_NS_8AttnArgsE"] == 128
    assert regs["_ZN3tfl11attn_kernelILi32EEEv14CUtensorMap_stS1_NS_8AttnArgsE"] == 120


def test_check_accepts_exactly_128():
    b.check_launch_registers(LOG.format(r64=128, r32=128))


@pytest.mark.parametrize("r64,r32", [(120, 128), (128, 96), (168, 128)])
def test_check_refuses_any_other_count(r64, r32):
    with pytest.raises(RuntimeError, match="setmaxnreg"):
        b.check_launch_registers(LOG.format(r64=r64, r32=r32))


def test_check_refuses_a_log_without_the_kernels():
    with pytest.raises(RuntimeError, match="no register count"):
        b.check_launch_registers("ptxas info    : Used 32 registers, used 0 barriers\n")


def test_the_built_attention_object_passes(tmp_path):
    # compile attention.cu as the build does and run the check on its log
    import subprocess
    out = tmp_path / "attention.o"
    cmd = [b._nvcc(), *b.ARCH, *b.FLAGS, "-Xptxas", "-v", "-c", f"{b.CSRC}/attention.cu", "-o", str(out)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    b.check_launch_registers(r.stdout + r.stderr)
