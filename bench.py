"""Benchmark: forward tokens/s of the Transformer-stack forward on one GB300.

Default workload: the largest single-GPU shape of the workload table,
B=32, S=100000, d_model=1024, H=16 (head_dim 64), d_ff=4096, 1 layer, causal,
full lengths (seed 0); --workload N picks another row of the table.
A step is one whole forward (all layers) over that batch; tokens per step =
B*S (every position, as the pages count tokens).

Prints ONE JSON line (rank 0).  Keys beyond the base contract:
  roofline      dominant kernel of the step: algorithmic work per launch /
                its CUDA-event duration, against the measured peak
  cpu_baseline  the fp64 oracle timed on this host on a bounded sample
  e2e           tokens/s from pinned host x / out, host<->device traffic inside
                the timed region: tfl_forward_host (the kernels read x and write
                out across the host link) or, for inputs over 4 GB,
                tfl_forward_streamed (batch slices of a thirty-second of the batch,
                their copies overlapping the forward of other slices)
  clocks        SM clock samples taken during the timed region
With --impl reference the fp64 oracle itself is timed as the reference arm.
Multi-GPU (torchrun): every rank runs an independent replica on its own
batch (sequences are independent; no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
# ex2.approx.f32 results per clock per SM, measured on GB300 with
# tests/probes/ex2_rate.cu (32.0 at 8 and 32 warps per SM)
MUFU_PER_CLK_PER_SM = 32


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, pg, device) -> float:
    """The largest of every rank's x (the job is as slow as its slowest rank); x itself
    without a process group.  device: where the reduction tensor lives (cuda for NCCL,
    cpu for gloo)."""
    if pg is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def replica_seed(rank: int) -> int:
    """Seed of the batch a rank runs: every rank an independent replica with its own
    batch (sequences are independent, so ranks exchange nothing on the data path)."""
    return rank


def job_value(world: int, units_per_rank: float, seconds: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return world * units_per_rank / seconds


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "tc_tflops": float(d["bf16_tflops"]),
                "tc_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "sm_max_mhz": float(d.get("sm_max_mhz", 2070.0)), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "tc_tflops": 1900.0, "tc_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0,
                "source": "fallback"}


class ClockSampler:
    """nvidia-smi SM clock / throttle sampling in the background."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path: str = ""):
        import tempfile
        self.idx = gpu_index
        self.proc = None
        self.path = path or os.path.join(tempfile.gettempdir(), f"tfl_clocks_gpu{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm), "reasons": sorted(reasons)}


def workload(idx: int) -> synth.Shape:
    return synth.WORKLOADS[idx]


def custom_shape(spec: str) -> synth.Shape:
    """'B,S,D,H,F,L,causal[,len_lo,len_hi]' -> a Shape (for small profiling cases)."""
    f = [int(v) for v in spec.split(",")]
    if len(f) not in (7, 9):
        raise SystemExit("--shape wants B,S,D,H,F,L,causal[,len_lo,len_hi]")
    lo, hi = (f[7], f[8]) if len(f) == 9 else (None, None)
    name = f"B{f[0]}_S{f[1]}_D{f[2]}_H{f[3]}_F{f[4]}_L{f[5]}_" + ("causal" if f[6] else "keymask")
    return synth.Shape(f[0], f[1], f[2], f[3], f[4], f[5], bool(f[6]), lo, hi, name=name)


def algorithmic(shape: synth.Shape, lens: np.ndarray, causal: bool):
    """Per-forward algorithmic FLOPs and per-kernel units (valid rows, allowed pairs only)."""
    D, F, H, L = shape.d_model, shape.d_ff, shape.n_heads, shape.n_layers
    hd = D // H
    lens = lens.astype(np.float64)
    valid = float(lens.sum())
    pairs = float((lens * (lens + 1) / 2).sum()) if causal else float((lens * lens).sum())
    lin = 2.0 * valid * (3 * D * D + D * D + 2 * D * F) * L
    att = 4.0 * pairs * hd * H * L
    return {"valid_tokens": valid, "pairs": pairs, "linear_flops": lin, "attn_flops": att,
            "attn_exps_per_launch": pairs * H, "attn_flops_per_launch": 4.0 * pairs * hd * H}


def gemm_flops(kind: str, shape: synth.Shape, valid: float):
    """Algorithmic FLOPs of one launch of a projection GEMM (valid rows only)."""
    D, F = shape.d_model, shape.d_ff
    nk = {"gemm_qkv": (3 * D, D), "gemm_oproj": (D, D), "gemm_ffn1": (F, D), "gemm_ffn2": (D, F)}.get(kind)
    return None if nk is None else 2.0 * valid * nk[0] * nk[1]


def kernel_bytes(kind: str, shape: synth.Shape, valid: float):
    """Algorithmic HBM bytes per launch of the row-streaming kernels (valid rows only;
    default precision: GEMM activations carry an fp16 hi plane and, in the same bytes as an fp16
    lo plane, its lo plane or its two e4m3 planes)."""
    D, F, L = shape.d_model, shape.d_ff, shape.n_layers
    # the fused chain (d_model 128), averaged over the forward's L launches: attention output
    # in, residual in, then either residual out + the next layer's qkv (fp16; its QKV
    # projection runs in the chain's tail) or, for the last layer, the fp32 model output
    chain = (L - 1) * (D * 2 + D * 4 + D * 4 + 3 * D * 2) + (D * 2 + D * 4 + D * 4)
    return {
        "gemm_qkv": valid * (2 * D * 2 + 3 * D * 2),
        "gemm_ffn1": valid * (D * 2 + F * 2),
        "gemm_oproj": valid * (D * 2 + D * 4 + D * 4 + D * 2),
        "gemm_ffn2": valid * (F * 2 + D * 4 + D * 4 + D * 2),
        "rownorm": valid * (D * 4 + 2 * D * 2),
        "postchain": valid * chain / L,
    }.get(kind)


def forward_bytes(shape: synth.Shape, valid: float):
    """Algorithmic HBM bytes of one forward under this implementation's kernel split
    (each intermediate written once and read once at its stored width, valid rows only)."""
    D, L = shape.d_model, shape.n_layers
    attn = valid * (3 * D * 2 + D * 2)  # q, k, v in; o out
    if D == 128 and shape.S <= 128 and shape.n_heads == 4 and L <= 8:  # the whole-stack kernel
        return stack_bytes(shape, valid)
    if D == 128:  # input LN, layer 0's QKV GEMM, then attention + fused chain per layer
        return (kernel_bytes("rownorm", shape, valid) + kernel_bytes("gemm_qkv", shape, valid)
                + L * (attn + kernel_bytes("postchain", shape, valid)))
    per_layer = (kernel_bytes("gemm_qkv", shape, valid) + attn + kernel_bytes("gemm_oproj", shape, valid)
                 + kernel_bytes("gemm_ffn1", shape, valid) + kernel_bytes("gemm_ffn2", shape, valid))
    return kernel_bytes("rownorm", shape, valid) + L * per_layer


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu
# capture of the benchmark workload (summaries in profiles/).  A figure is valid
# only while every kernel source it was taken with is unchanged: the fingerprint is
# the sha256 prefix over all files of the package's csrc/ directory; otherwise
# traffic is reported null.
# The translation unit of each measured kernel plus every kernel header: the
# fingerprint a traffic figure was captured with (host code such as api.cu is
# not part of any kernel's build).
KERNEL_SOURCES = {
    "stack": ["stack.cu"],
    "postchain": ["postchain.cu"],
    "attention": ["attention.cu"],
    "gemm_qkv": ["gemm.cu"],
    "gemm_oproj": ["gemm.cu"],
    "gemm_ffn1": ["gemm.cu"],
    "gemm_ffn2": ["gemm.cu"],
}
KERNEL_HEADERS = ["kernels.h", "ptx.cuh", "mathfn.cuh", "xpose.cuh", "chainops.cuh"]

NCU_TRAFFIC = {
    # (kernel, workload): (kernel source fingerprint, bytes per launch); entries whose
    # fingerprint no longer matches the sources report null
    ("postchain", "B64_S1024_D128_causal_ragged"): ("3308ef9bf974", 42.620416e6 + 29.589504e6),
    ("stack", "B2048_S128_D128_H4_F512_L4_keymask"): ("ee76cb851076", 87.525632e6 + 86.630912e6),  # lengths U[32,128]
    ("attention", "B2_S16384_D1024_H16_F4096_L1_causal"): ("82bcd7cfdc72", 209.170944e6 + 49.693184e6),
    ("gemm_qkv", "B16_S512_D1024_H4_causal"): ("f4a5a3a4c7ff", 46.386176e6 + 11.332864e6),
    ("gemm_oproj", "B16_S512_D1024_H4_causal"): ("f4a5a3a4c7ff", 54.558976e6 + 2.426624e6),
    ("gemm_ffn1", "B16_S512_D1024_H4_causal"): ("f4a5a3a4c7ff", 51.184384e6 + 86.635264e6),
    ("gemm_ffn2", "B16_S512_D1024_H4_causal"): ("f4a5a3a4c7ff", 185.78688e6 + 18.534912e6),
}


def csrc_fingerprint(kernel: str = None) -> str:
    """sha256 prefix over the package's csrc/ files (all of them, or one kernel's sources)."""
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "attention_qkv_gemm_gb300", "csrc")
    files = sorted(os.listdir(d)) if kernel is None else sorted(KERNEL_SOURCES[kernel] + KERNEL_HEADERS)
    for f in files:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:12]


# Workloads too large to capture under ncu take a smaller case's DRAM bytes per launch,
# scaled by the tokens a launch processes (the kernel reads q, k, v and writes o once per
# token; its keys and values are re-read from L2, not HBM, under the grouped work order):
# (kernel, workload): (captured workload, tokens captured, tokens of the full launch)
NCU_TRAFFIC_SCALED = {
    ("attention", "B32_S100000_D1024_H16_causal"): ("B2_S16384_D1024_H16_F4096_L1_causal", 2 * 16384, 32 * 100000),
    ("stack", "B10000_S128_D128_keymask_ragged"): ("B2048_S128_D128_H4_F512_L4_keymask", 2048 * 128, 10000 * 128),
}


def ncu_traffic(kernel: str, workload: str):
    if (kernel, workload) in NCU_TRAFFIC_SCALED:
        src, t_small, t_full = NCU_TRAFFIC_SCALED[(kernel, workload)]
        small = ncu_traffic(kernel, src)
        return None if small is None else small * t_full / t_small
    e = NCU_TRAFFIC.get((kernel, workload))
    if e is None or kernel not in KERNEL_SOURCES:
        return None
    sha, nbytes = e
    return nbytes if csrc_fingerprint(kernel) == sha else None


def ncu_traffic_note(kernel: str, workload: str):
    if (kernel, workload) in NCU_TRAFFIC_SCALED:
        src, t_small, t_full = NCU_TRAFFIC_SCALED[(kernel, workload)]
        return f"ncu DRAM bytes of a {src} launch scaled by tokens ({t_full}/{t_small})"
    return None


def live_tiles(shape: synth.Shape, lens: np.ndarray) -> int:
    """128-row tiles of the flattened [B*S] token axis that the kernels process: those
    holding a valid row or a padding row read as a key (rows below len_b rounded up to
    64, at most S)."""
    S, n = shape.S, 0
    M = shape.B * S
    for t in range((M + 127) // 128):
        m0, m1 = t * 128, min(M, t * 128 + 128)
        for b in range(m0 // S, (m1 - 1) // S + 1):
            kr = min(S, (int(lens[b]) + 63) // 64 * 64)
            if max(m0, b * S) < min(m1, b * S + kr):
                n += 1
                break
    return n


def chain_executed_flops(shape: synth.Shape, lens: np.ndarray) -> float:
    """Tensor FLOPs the fused chain (d_model 128) executes per forward: per live 128-row
    tile, 128x128x16 MMAs -- o_proj 16 (8 k-steps, weight hi and lo), FFN-in and FFN-out
    24 per 128-wide d_ff chunk each (operand and weight split, 3 MMAs per k-step), and the
    next layer's QKV projection 72 in every launch but the last."""
    L, nch = shape.n_layers, shape.d_ff // 128
    mmas = L * (16 + 48 * nch) + (L - 1) * 72
    return float(live_tiles(shape, lens)) * mmas * 2.0 * 128 * 128 * 16


def stack_executed_flops(shape: synth.Shape, lens: np.ndarray) -> float:
    """Tensor FLOPs the whole-stack kernel executes per forward, in 128x128x16 MMA
    equivalents per sequence (one 128-row tile) and layer: QKV 72 (3 blocks x 8
    k-steps x 3 split MMAs), attention per head S 2 + P V 2 (N = 32) + row sum 1 (N = 16),
    o_proj 16, FFN 48 per 128-wide d_ff chunk."""
    nch = shape.d_ff // 128
    per_layer = 72 + (shape.n_heads * 5) + 16 + 48 * nch
    seqs = int((lens > 0).sum())
    return float(seqs) * shape.n_layers * per_layer * 2.0 * 128 * 128 * 16


def stack_bytes(shape: synth.Shape, valid: float) -> float:
    """Algorithmic HBM bytes of the whole-stack kernel per forward: x of the valid rows in,
    every output row out (fp32), and the packed fp16 weights (hi and lo) once."""
    D, F, L = shape.d_model, shape.d_ff, shape.n_layers
    return valid * D * 4 + shape.B * shape.S * D * 4 + L * (4 * D * D + 2 * D * F) * 2 * 2


# Sequences longer than this are sampled by query rows for the oracle timing (one
# causal layer: a row depends only on the keys before it, so a row sample is exact)
ORACLE_FULL_S = 8192
ORACLE_ROWS = 64


def oracle_rows(shape):
    if shape.S <= ORACLE_FULL_S or not (shape.causal and shape.n_layers == 1):
        return None
    rng = np.random.default_rng(12345)
    return np.unique(np.concatenate([[0, shape.S - 1], rng.choice(shape.S, ORACLE_ROWS - 2, replace=False)]))


def run_oracle_sample(shape, prm, seed, n_seq):
    """Time the fp64 oracle on n_seq sequences (or on a row sample of them); returns
    (seconds, output rows computed)."""
    import oracle
    lens = synth.lengths(seed, shape)
    batches = np.arange(n_seq)
    x = synth.input_x(seed, shape, batches=batches)
    rows = oracle_rows(shape)
    t0 = time.perf_counter()
    oracle.forward(prm, shape.n_heads, x, lens[batches], shape.causal, rows=rows)
    dt = time.perf_counter() - t0
    return dt, n_seq * (shape.S if rows is None else len(rows))


def oracle_sample_text(shape, n_seq, tok):
    rows = oracle_rows(shape)
    if rows is None:
        return f"{n_seq} of {shape.B} sequences ({tok} tokens), fp64 numpy"
    return (f"{n_seq} of {shape.B} sequences x {len(rows)} sampled query rows ({tok} output rows; keys and values "
            f"projected for every position up to the last sampled row), fp64 numpy")


def reference_arm(args, shape, world, rank):
    """The fp64 oracle timed as the reference arm (host cores, bounded sample per step)."""
    if rank != 0:
        return 0
    prm = synth.params(0, shape)
    n_seq = max(1, min(shape.B, args.ref_seqs if oracle_rows(shape) is None else 1))
    for _ in range(max(0, min(args.warmup, 1))):
        run_oracle_sample(shape, prm, 0, 1)
    times = []
    tok = 0
    for _ in range(args.steps):
        dt, tok = run_oracle_sample(shape, prm, 0, n_seq)
        times.append(dt)
    ms = 1e3 * statistics.mean(times)
    value = tok / (ms / 1e3)
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": "forward_tokens_per_s", "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(shape),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": oracle_sample_text(shape, n_seq, tok) + " per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def compute_dtype(shape) -> str:
    """Arithmetic types of the path: fp16 tensor-core products on split operands (fp32
    accumulation and fp32 row work), plus e4m3 products for the split GEMMs' correction terms
    above d_model 128 (the library's default fp8_corrections)."""
    return "f16+e4m3" if shape.d_model > 128 else "f16"


def e2e_slice(shape, arg: int) -> int:
    """Sequences per slice of the streamed end-to-end path: 0 (no slicing: tfl_forward_host)
    unless the fp32 input is over 4 GB, else a thirty-second of the batch (at least one
    sequence): small slices keep the copies that nothing overlaps (the first slice in, the last
    one out) short; arg > 0 forces a slice size, arg < 0 turns slicing off."""
    if arg < 0:
        return 0
    if arg > 0:
        return min(arg, shape.B)
    return 0 if shape.B * shape.S * shape.d_model * 4 <= (4 << 30) else max(1, shape.B // 32)


def config_dict(shape):
    return {"workload": shape.name, "B": shape.B, "S": shape.S, "d_model": shape.d_model, "n_heads": shape.n_heads,
            "d_ff": shape.d_ff, "n_layers": shape.n_layers, "causal": shape.causal,
            "lengths": "full" if shape.len_lo is None else f"uniform[{shape.len_lo},{shape.len_hi}]",
            "l2": "flushed (256 MiB write) between timed steps", "seed": 0}


# An instrumented copy of the forward attention kernel for --attn-cycles (profiling only):
# clock64 counters around each wait and each issue sequence of the two MMA-issuing threads, and
# around the softmax warps' wait for S and their sub-block loop, summed per role into a device
# array that tfl_attn_cycles_fetch reads and clears.  The copy is made from csrc/attention.cu at
# run time by inserting text at fixed anchors (each must occur exactly once, or the mode stops),
# and built into a separate library under _build/cycles/ that nothing else loads.
# Slots: 0-4 P V thread (total, waiting for P, waiting for the K/V stage, issuing MMAs and
# commits, sub-blocks), 8-12 the same for the Q K^T thread (its first wait is for P V of the
# buffer's previous sub-block), 5-7 softmax warps (total, waiting for S, the sub-block loop),
# 13 softmax warps' output phase.
ATTN_CYCLE_PATCHES = [
    ("namespace tfl {\n",
     "namespace tfl {\n__device__ unsigned long long g_attn_cycles[16];\n"),
    ("    bool first_item = true, ok = true;\n",
     "    bool first_item = true, ok = true;\n"
     "    long long cy_w = 0, cy_kv = 0, cy_is = 0, cy_n = 0;\n"
     "    const long long cy_t0 = clock64();\n"),
    ("        if (is_qk) {\n          // S[b] last held",
     "        const long long cy_a = clock64();\n        if (is_qk) {\n          // S[b] last held"),
    ("        if (h == 0) {\n          if (!wait_bounded(&kv_full[st], kvph, wc)) {",
     "        const long long cy_b = clock64();\n        cy_w += cy_b - cy_a;\n"
     "        if (h == 0) {\n          if (!wait_bounded(&kv_full[st], kvph, wc)) {"),
    ("        tc_fence_after();\n        mma_issued = true;\n",
     "        const long long cy_c = clock64();\n        cy_kv += cy_c - cy_b;\n"
     "        tc_fence_after();\n        mma_issued = true;\n"),
    ("        if (stage_done) {\n          if (++st == C::NST) {",
     "        cy_is += clock64() - cy_c;\n        if (stage_done) {\n          if (++st == C::NST) {"),
    ("      g += nsub;\n",
     "      g += nsub;\n      cy_n += nsub;\n"),
    ("      if (++qb_i == C::NQ) qb_i = 0;\n    }\n   }\n  }\n  } else {",
     "      if (++qb_i == C::NQ) qb_i = 0;\n    }\n"
     "    {\n      const int cy_o = is_qk ? 8 : 0;\n"
     "      atomicAdd(&g_attn_cycles[cy_o + 0], (unsigned long long)(clock64() - cy_t0));\n"
     "      atomicAdd(&g_attn_cycles[cy_o + 1], (unsigned long long)cy_w);\n"
     "      atomicAdd(&g_attn_cycles[cy_o + 2], (unsigned long long)cy_kv);\n"
     "      atomicAdd(&g_attn_cycles[cy_o + 3], (unsigned long long)cy_is);\n"
     "      atomicAdd(&g_attn_cycles[cy_o + 4], (unsigned long long)cy_n);\n    }\n"
     "   }\n  }\n  } else {"),
    ("    uint8_t* xst = sX + (warp - 4) * C::XPW;\n",
     "    uint8_t* xst = sX + (warp - 4) * C::XPW;\n"
     "    long long cy_s = 0, cy_body = 0, cy_out = 0;\n"
     "    const long long cy_t0 = clock64();\n"),
    ("        if (!wait_bounded(&s_full[gg % 3u], (gg / 3u) & 1u, wc)) return false;\n",
     "        const long long cy_a = clock64();\n"
     "        if (!wait_bounded(&s_full[gg % 3u], (gg / 3u) & 1u, wc)) return false;\n"
     "        cy_s += clock64() - cy_a;\n"),
    ("      int u = 0;\n      for (; ok && u < nfull; ++u, ++g) ok = body(std::true_type{}, u);\n"
     "      for (; ok && u < nsub; ++u, ++g) ok = body(std::false_type{}, u);\n",
     "      int u = 0;\n      const long long cy_b = clock64();\n"
     "      for (; ok && u < nfull; ++u, ++g) ok = body(std::true_type{}, u);\n"
     "      for (; ok && u < nsub; ++u, ++g) ok = body(std::false_type{}, u);\n"
     "      cy_body += clock64() - cy_b;\n      const long long cy_o = clock64();\n"),
    ("      if (lane == 0) mbar_arrive(o_empty);\n    }\n  }\n\n  // ---",
     "      if (lane == 0) mbar_arrive(o_empty);\n      cy_out += clock64() - cy_o;\n    }\n"
     "    if (lane == 0) {\n"
     "      atomicAdd(&g_attn_cycles[5], (unsigned long long)(clock64() - cy_t0));\n"
     "      atomicAdd(&g_attn_cycles[6], (unsigned long long)cy_s);\n"
     "      atomicAdd(&g_attn_cycles[7], (unsigned long long)cy_body);\n"
     "      atomicAdd(&g_attn_cycles[13], (unsigned long long)cy_out);\n    }\n  }\n\n  // ---"),
    ("}  // namespace tfl\n",
     "}  // namespace tfl\n\n"
     "extern \"C\" int tfl_attn_cycles_fetch(unsigned long long* out) {\n"
     "  cudaError_t e = cudaMemcpyFromSymbol(out, tfl::g_attn_cycles, 16 * sizeof(unsigned long long));\n"
     "  static const unsigned long long zero[16] = {0};\n"
     "  if (e == cudaSuccess) e = cudaMemcpyToSymbol(tfl::g_attn_cycles, zero, sizeof(zero));\n"
     "  return (int)e;\n}\n"),
]


def attention_cycles_source(src: str) -> str:
    """attention.cu with the --attn-cycles counters inserted (every anchor exactly once)."""
    for anchor, repl in ATTN_CYCLE_PATCHES:
        n = src.count(anchor)
        if n != 1:
            raise RuntimeError(f"--attn-cycles: an anchor occurs {n} times in attention.cu "
                               f"(the kernel changed; update ATTN_CYCLE_PATCHES): {anchor[:60]!r}")
        src = src.replace(anchor, repl)
    return src


def build_attention_cycles_lib() -> str:
    """Compile the instrumented attention copy and link it with the library's other objects into
    _build/cycles/libtfl_cycles.so; the same launch-register check as the library build."""
    from attention_qkv_gemm_gb300 import build as libbuild
    libbuild.build()
    out = os.path.join(libbuild.BUILD, "cycles")
    os.makedirs(out, exist_ok=True)
    with open(os.path.join(libbuild.CSRC, "attention.cu")) as f:
        src = attention_cycles_source(f.read())
    cu, obj, lib = (os.path.join(out, n) for n in ("attention_cycles.cu", "attention_cycles.o",
                                                  "libtfl_cycles.so"))
    with open(cu, "w") as f:
        f.write(src)
    nvcc = libbuild._nvcc()
    r = subprocess.run([nvcc, *libbuild.ARCH, *libbuild.FLAGS, "-Xptxas", "-v", "-c", cu, "-o", obj],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on the instrumented attention:\n{r.stdout}\n{r.stderr}")
    libbuild.check_launch_registers(r.stdout + r.stderr)
    objs = [os.path.join(libbuild.BUILD, os.path.splitext(s)[0] + ".o") for s in libbuild.SOURCES
            if s != "attention.cu"]
    r = subprocess.run([nvcc, *libbuild.ARCH, "-shared", "-o", lib, obj, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return lib


def attention_cycles_report(c, B, S, H, hd, causal, launches):
    """Cycles per 64-key sub-block and CTA for each role, from the summed counter slots of the
    instrumented attention copy (see ATTN_CYCLE_PATCHES)."""
    n_pv, n_qk = c[4], c[12]  # sub-blocks summed over the CTAs (each issuer sees every sub-block)
    warps = 4.0 * n_pv        # the softmax counters are summed over the four warps of each CTA: per warp
    per = lambda v, n: round(v / n, 1) if n else None
    line = {"metric": "attention_cycles_per_subblock", "unit": "SM cycles per 64-key sub-block and CTA",
            "config": {"B": B, "S": S, "n_heads": H, "head_dim": hd, "causal": bool(causal), "launches": launches},
            "pv_thread": {"total": per(c[0], n_pv), "waiting_for_p": per(c[1], n_pv),
                          "waiting_for_kv": per(c[2], n_pv), "issuing": per(c[3], n_pv)},
            "qk_thread": {"total": per(c[8], n_qk), "waiting_for_pv": per(c[9], n_qk),
                          "waiting_for_kv": per(c[10], n_qk), "issuing": per(c[11], n_qk)},
            "softmax_warp": {"total": per(c[5], warps), "waiting_for_s": per(c[6], warps),
                             "subblock_loop": per(c[7], warps), "output": per(c[13], warps)},
            "note": "instrumented copy of attention.cu (clock64 around each wait and issue sequence); "
                    "the counters slow the kernel a few per cent"}
    return line


def attention_cycles_bench(args):
    """The forward attention kernel's cycles per 64-key sub-block and CTA, per role, from the
    instrumented copy (B,S,H,head_dim,causal; one warm-up launch, then --steps launches)."""
    import ctypes
    import torch
    import attention_qkv_gemm_gb300 as pkg
    B, S, H, hd, causal = [int(v) for v in args.attn_cycles.split(",")]
    lib = pkg.load(build_attention_cycles_lib())
    buf = (ctypes.c_ulonglong * 16)()
    D = H * hd
    g = torch.Generator(device="cuda").manual_seed(0)
    qkv = torch.randn(B, S, 3 * D, device="cuda", generator=g).half()
    o = torch.empty(B, S, D, device="cuda", dtype=torch.float16)
    lse = torch.empty(B, H, S, device="cuda", dtype=torch.float32)
    a = pkg.tfl_attn_create(B, S, H, hd)
    sp = torch.cuda.current_stream().cuda_stream
    fwd = lambda: pkg.tfl_attn_forward(a, qkv.data_ptr(), None, causal, o.data_ptr(), lse.data_ptr(), sp)
    fwd()
    torch.cuda.synchronize()
    if lib.tfl_attn_cycles_fetch(buf) != 0:
        raise RuntimeError("tfl_attn_cycles_fetch failed")
    for _ in range(args.steps):
        fwd()
    torch.cuda.synchronize()
    if pkg.tfl_attn_status(a, sp) != 0:
        raise RuntimeError(pkg.tfl_last_error())
    if lib.tfl_attn_cycles_fetch(buf) != 0:
        raise RuntimeError("tfl_attn_cycles_fetch failed")
    pkg.tfl_attn_destroy(a)
    print(json.dumps(attention_cycles_report([float(v) for v in buf], B, S, H, hd, causal, args.steps)))


def attention_backward_bench(args):
    """Standalone attention (tfl_attn_forward / tfl_attn_backward) on random fp16 q, k, v and
    dO of the given shape: CUDA-event time of each, against the dense tensor peak.
    Algorithmic FLOPs per allowed (query, key) pair and head: forward 4 hd (Q K^T, P V),
    backward 10 hd (Q K^T rebuilt, dO V^T, P^T dO, dS K, dS^T Q)."""
    import torch
    import attention_qkv_gemm_gb300 as pkg
    from attention_qkv_gemm_gb300 import build as libbuild
    B, S, H, hd, causal = [int(v) for v in args.attn_bwd.split(",")]
    libbuild.build()
    pkg.load()
    D = H * hd
    g = torch.Generator(device="cuda").manual_seed(0)
    qkv = torch.randn(B, S, 3 * D, device="cuda", generator=g).half()
    dout = torch.randn(B, S, D, device="cuda", generator=g).half()
    o = torch.empty(B, S, D, device="cuda", dtype=torch.float16)
    lse = torch.empty(B, H, S, device="cuda", dtype=torch.float32)
    dqkv = torch.empty(B, S, 3 * D, device="cuda", dtype=torch.float32)
    a = pkg.tfl_attn_create(B, S, H, hd)
    st = torch.cuda.current_stream()
    sp = st.cuda_stream
    fwd = lambda: pkg.tfl_attn_forward(a, qkv.data_ptr(), None, causal, o.data_ptr(), lse.data_ptr(), sp)
    bwd = lambda: pkg.tfl_attn_backward(a, qkv.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(), None,
                                        causal, dqkv.data_ptr(), sp)
    for _ in range(args.warmup):
        fwd()
        bwd()
    if pkg.tfl_attn_status(a, sp) != 0:
        raise RuntimeError(pkg.tfl_last_error())
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    for e in ev:
        e[0].record(st)
        fwd()
        e[1].record(st)
        bwd()
        e[2].record(st)
    torch.cuda.synchronize()
    if pkg.tfl_attn_status(a, sp) != 0:
        raise RuntimeError(pkg.tfl_last_error())
    pkg.tfl_attn_destroy(a)
    f_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    b_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    pairs = B * (S * (S + 1) / 2 if causal else S * S)
    peaks = load_peaks()
    ff, bf = 4.0 * hd * pairs * H, 10.0 * hd * pairs * H
    line = {"metric": "attention_backward_tflops", "value": bf / (b_ms / 1e3) / 1e12, "unit": "TFLOP/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": f_ms + b_ms,
            "higher_is_better": True, "dtype": "f16", "data": "synthetic",
            "config": {"workload": f"attention B{B} S{S} H{H} hd{hd} " + ("causal" if causal else "full"),
                       "B": B, "S": S, "n_heads": H, "head_dim": hd, "causal": bool(causal)},
            "forward_ms": f_ms, "backward_ms": b_ms,
            "roofline": {"bound": "tensor", "peak": peaks["tc_tflops"], "unit": "TFLOP/s",
                         "forward": {"achieved": ff / (f_ms / 1e3) / 1e12,
                                     "frac": ff / (f_ms / 1e3) / 1e12 / peaks["tc_tflops"]},
                         "backward": {"achieved": bf / (b_ms / 1e3) / 1e12,
                                      "frac": bf / (b_ms / 1e3) / 1e12 / peaks["tc_tflops"]},
                         "note": "FLOPs per allowed pair and head: forward 4 hd, backward 10 hd"}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=4,
                    help="index into the workload table (default: B32 S100000, the largest)")
    ap.add_argument("--shape", default="", help="B,S,D,H,F,L,causal[,len_lo,len_hi]: a custom (profiling) shape")
    ap.add_argument("--clocks-csv", default="", help="where to keep the nvidia-smi clock samples")
    ap.add_argument("--ref-seqs", type=int, default=2, help="sequences per reference/oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-slice", type=int, default=0,
                    help="sequences per slice of the streamed e2e path (0: automatic, <0: off)")
    ap.add_argument("--whole-stack", type=int, default=1,
                    help="tfl_options.whole_stack: 1 (default) or 0 (per-layer kernels)")
    ap.add_argument("--attn-bwd", default="",
                    help="B,S,H,head_dim,causal: time the standalone attention forward + backward instead")
    ap.add_argument("--attn-cycles", default="",
                    help="B,S,H,head_dim,causal: cycles per sub-block of the forward attention kernel's roles, "
                         "from an instrumented copy (profiling)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup

    world, rank, local = dist_env()
    if args.attn_bwd and args.impl == "ours":
        return attention_backward_bench(args)
    if args.attn_cycles and args.impl == "ours":
        return attention_cycles_bench(args)
    shape = custom_shape(args.shape) if args.shape else workload(args.workload)
    if args.impl == "reference":
        return reference_arm(args, shape, world, rank)

    import torch
    import attention_qkv_gemm_gb300 as pkg
    from attention_qkv_gemm_gb300 import build as libbuild

    torch.cuda.set_device(local)
    n_sms = torch.cuda.get_device_properties(local).multi_processor_count
    if rank == 0 or world == 1:
        libbuild.build()
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
        dist.barrier()
        libbuild.build()
    pkg.load()

    seed = replica_seed(rank)
    prm = synth.params(seed, shape)
    lens_np = synth.lengths(seed, shape)
    x_np = synth.input_x(seed, shape)
    dev = torch.device("cuda", local)
    x = torch.from_numpy(x_np).to(dev)
    # the pinned host copy for the e2e leg, made now so that the numpy array can go (host
    # memory per rank: the pinned input and output, 26 GB at B32 S100000)
    hx = torch.from_numpy(x_np).pin_memory()
    del x_np
    lens = torch.from_numpy(lens_np).to(dev)
    out = torch.empty_like(x)
    opts = pkg.tfl_default_options()
    opts.whole_stack = args.whole_stack
    m = pkg.TransformerStack(shape.B, shape.S, shape.d_model, shape.n_heads, shape.d_ff, shape.n_layers, prm,
                             options=opts)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def fwd():
        pkg.tfl_forward(m.handle, x.data_ptr(), lens.data_ptr(), int(shape.causal), out.data_ptr(), sp)

    for _ in range(args.warmup):
        fwd()
    rc = m.status(sp)
    if rc != 0:
        raise RuntimeError(f"device status {rc}: {pkg.tfl_last_error()}")

    # ---------------- timed region: graph replays, L2 flushed between steps
    sampler = ClockSampler(local, args.clocks_csv)
    sampler.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    for s, e in evs:
        flush.fill_(1.0)
        s.record(stream)
        fwd()
        e.record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    step_ms = [s.elapsed_time(e) for s, e in evs]
    clocks = sampler.stop()
    rc = m.status(sp)
    if rc != 0:
        raise RuntimeError(f"device status {rc}: {pkg.tfl_last_error()}")
    ms = max_over_ranks(statistics.mean(step_ms), pg, dev)
    tokens = shape.B * shape.S
    value = job_value(world, tokens, ms / 1e3)

    # ---------------- per-kernel times (eager, events around every launch)
    prof = {}
    for _ in range(3):
        for kind, kms in pkg.tfl_profile_forward(m.handle, x.data_ptr(), lens.data_ptr(), int(shape.causal),
                                                 out.data_ptr(), sp):
            prof.setdefault(kind, []).append(kms)
    per_kind = {k: (sum(v) / 3.0, len(v) // 3) for k, v in prof.items()}  # ms per forward, launches per forward
    dom = max(per_kind, key=lambda k: per_kind[k][0])
    dom_ms_launch = per_kind[dom][0] / per_kind[dom][1]
    alg = algorithmic(shape, lens_np, shape.causal)
    peaks = load_peaks()
    # a launch longer than this runs under the power cap: the sustained tensor peak applies
    tc_peak = peaks["tc_tflops_sustained"] if dom_ms_launch > 50.0 else peaks["tc_tflops"]
    if dom == "attention":
        exps = alg["attn_exps_per_launch"]
        fl = alg["attn_flops_per_launch"]
        mufu_peak = MUFU_PER_CLK_PER_SM * n_sms * peaks["sm_max_mhz"] * 1e6 / 1e9
        mufu = exps / (dom_ms_launch / 1e3) / 1e9
        tflops = fl / (dom_ms_launch / 1e3) / 1e12
        # the unit that bounds the launch at peak: one exp2 per allowed (query, key) pair and
        # head against 4 * head_dim tensor FLOPs for the same pair (QK^T and P V)
        if exps / (mufu_peak * 1e9) >= fl / (tc_peak * 1e12):
            roof = {"kernel": "attention", "bound": "alu", "achieved": mufu, "peak": mufu_peak, "unit": "Gexp2/s",
                    "frac": mufu / mufu_peak, "tensor_tflops": tflops}
        else:
            roof = {"kernel": "attention", "bound": "tensor", "achieved": tflops, "peak": tc_peak,
                    "unit": "TFLOP/s", "frac": tflops / tc_peak, "mufu_gexp2_s": mufu, "mufu_frac": mufu / mufu_peak}
        roof["traffic"] = ncu_traffic("attention", shape.name)
        roof["note"] = (f"MUFU ex2 rate: 32/clk/SM (measured) x {n_sms} SMs x max SM clock; per launch = allowed "
                        "(query, key) pairs x heads; tensor = 4 x head_dim FLOPs per allowed pair and head")
    elif dom == "stack":
        # the whole forward in one launch: algorithmic FLOPs against the dense tensor peak, and
        # the split-operand MMAs it executes; HBM moves only x, the output and the weights
        fl = alg["linear_flops"] + alg["attn_flops"]
        achieved = fl / (dom_ms_launch / 1e3) / 1e12
        ex = stack_executed_flops(shape, lens_np)
        hb = stack_bytes(shape, alg["valid_tokens"])
        roof = {"kernel": "stack", "bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                "frac": achieved / tc_peak, "traffic": ncu_traffic("stack", shape.name),
                "algorithmic_flops_per_launch": fl,
                "tensor_executed": {"achieved": ex / (dom_ms_launch / 1e3) / 1e12, "peak": tc_peak,
                                    "unit": "TFLOP/s", "frac": ex / (dom_ms_launch / 1e3) / 1e12 / tc_peak,
                                    "executed_flops_per_launch": ex},
                "hbm": {"algorithmic_bytes_per_launch": hb, "achieved": hb / (dom_ms_launch / 1e3) / 1e9,
                        "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": hb / (dom_ms_launch / 1e3) / 1e9 / peaks["hbm_gbs"]},
                "note": "split-fp16 operands: the executed MMAs are 2-3x the algorithmic FLOPs"}
    elif shape.d_model > 128 and gemm_flops(dom, shape, alg["valid_tokens"]) is not None:
        # d_model > 128: the projection GEMMs are dense contractions (fp16 operands, fp32
        # accumulate), measured against the dense tensor peak (fp16 = bf16 nominal rate)
        fl = gemm_flops(dom, shape, alg["valid_tokens"])
        achieved = fl / (dom_ms_launch / 1e3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": tc_peak,
                "unit": "TFLOP/s", "frac": achieved / tc_peak, "traffic": ncu_traffic(dom, shape.name),
                "algorithmic_flops_per_launch": fl,
                "note": "split operands: per 16-wide k-step an fp16 product and two e4m3 correction products "
                        "at twice the fp16 rate (two fp16 MMAs' time; o_proj: two fp16 MMAs); achieved counts "
                        "the algorithmic 2*M*N*K only"}
    else:
        by = kernel_bytes(dom, shape, alg["valid_tokens"])
        achieved = by / (dom_ms_launch / 1e3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic(dom, shape.name),
                "algorithmic_bytes_per_launch": by}
        if dom == "postchain":
            # the split-operand MMAs the chain executes, against the tensor peak: the unit
            # that binds this kernel (see profiles/postchain_B64_S1024_D128.md)
            ex = chain_executed_flops(shape, lens_np) / shape.n_layers
            roof["tensor_executed"] = {"achieved": ex / (dom_ms_launch / 1e3) / 1e12, "peak": tc_peak,
                                       "unit": "TFLOP/s",
                                       "frac": ex / (dom_ms_launch / 1e3) / 1e12 / tc_peak,
                                       "executed_flops_per_launch": ex}
    note = ncu_traffic_note(dom, shape.name)
    if note and roof.get("traffic") is not None:
        roof["traffic_note"] = note
    roof["peak_source"] = peaks["source"] + (" (sustained)" if roof["unit"] == "TFLOP/s" and tc_peak != peaks["tc_tflops"] else "")
    roof["launch_ms"] = dom_ms_launch
    roof["kernels_ms_per_forward"] = {k: round(v[0], 4) for k, v in per_kind.items()}

    # ---------------- e2e from pinned host buffers, host<->device traffic inside the timed region
    hl = torch.from_numpy(lens_np).pin_memory()
    ho = torch.empty_like(hx).pin_memory()
    slice_b = e2e_slice(shape, args.e2e_slice)
    if slice_b:
        # batch slices streamed through a handle of the slice's batch size, copies of the
        # next and previous slices overlapping the forward of the current one
        ms_ = pkg.TransformerStack(slice_b, shape.S, shape.d_model, shape.n_heads, shape.d_ff, shape.n_layers, prm)

        def e2e_step():
            pkg.tfl_forward_streamed(ms_.handle, hx.data_ptr(), hl.data_ptr(), shape.B, int(shape.causal),
                                     ho.data_ptr(), sp)
            return pkg.tfl_status(ms_.handle, sp)
        e2e_path = f"tfl_forward_streamed, slices of {slice_b} sequences"
    else:
        ms_ = None

        def e2e_step():
            return pkg.tfl_forward_host(m.handle, hx.data_ptr(), hl.data_ptr(), int(shape.causal), ho.data_ptr(), sp)
        e2e_path = "tfl_forward_host (kernels read x and write out across the host link)"
    for _ in range(2):
        e2e_step()
    e2e_t = []
    for _ in range(max(3, min(args.steps, 10))):
        t0 = time.perf_counter()
        rc2 = e2e_step()
        e2e_t.append(time.perf_counter() - t0)
        if rc2 != 0:
            raise RuntimeError(f"e2e status {rc2}")
    if ms_ is not None:
        ms_.close()
    e2e_s = max_over_ranks(statistics.mean(e2e_t), pg, dev)
    e2e = {"value": job_value(world, tokens, e2e_s), "unit": "tokens/s", "h2d_bytes_per_step": int(hx.numel() * 4 + hl.numel() * 4),
           "d2h_bytes_per_step": int(ho.numel() * 4), "path": e2e_path, "ms_per_step": e2e_s * 1e3}

    launches = pkg.tfl_launch_count(m.handle, int(shape.causal)) * args.steps
    m.close()

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return 0

    # whole forward against its own bound: t_bound = max(HBM bytes / copy bandwidth,
    # algorithmic FLOPs / dense fp16 tensor peak), both measured peaks
    fb = forward_bytes(shape, alg["valid_tokens"])
    flops = alg["linear_flops"] + alg["attn_flops"]
    t_hbm, t_tc = fb / (peaks["hbm_gbs"] * 1e9), flops / (peaks["tc_tflops"] * 1e12)
    fwd_roof = {"bytes": fb, "flops": flops, "t_bound_ms": max(t_hbm, t_tc) * 1e3,
                "bound": "hbm" if t_hbm >= t_tc else "tensor", "frac": max(t_hbm, t_tc) / (ms / 1e3),
                "peak_source": peaks["source"]}

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        n_seq = min(shape.B, args.ref_seqs)
        dt, tok = run_oracle_sample(shape, prm, seed, n_seq)
        cpu = {"value": tok / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": oracle_sample_text(shape, n_seq, tok)}

    line = {
        "metric": "forward_tokens_per_s", "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": compute_dtype(shape), "data": "synthetic", "config": config_dict(shape), "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
        "algorithmic": {"valid_tokens": alg["valid_tokens"], "gflop": (alg["linear_flops"] + alg["attn_flops"]) / 1e9,
                        "tflops_achieved": (alg["linear_flops"] + alg["attn_flops"]) / (ms / 1e3) / 1e12,
                        "valid_tokens_per_s": job_value(world, alg["valid_tokens"], ms / 1e3)},
        "forward_roofline": fwd_roof,
    }
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
