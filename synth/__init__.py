"""Seeded synthetic inputs for the Transformer-stack forward.

This module is shared by the fp64 oracle and by the GPU path's tests and
benchmark.  It holds random-number generation and the workload table only:
none of the model's arithmetic lives here.

Generator: a counter-based normal sampler.  Every tensor gets its own stream
key, and element ``i`` of that stream is a pure function of (seed, stream, i),
so any slice can be produced without generating what comes before it.

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014) mixes the 64-bit counter.
* Box-Muller (1958) turns two 53-bit uniforms into one N(0, 1) draw, computed
  in float64 and rounded once to float32.

Workload shapes and value distributions follow the five benchmark shapes of
the TikTok TechJam 2026 "GPU Transformer Optimization" problem as restated in
the workload table below: x ~ N(0, 1); weights ~ N(0, 1/fan_in), i.e. standard
deviation 1/sqrt(fan_in); biases ~ N(0, 0.02) read as standard deviation 0.02;
LayerNorm gamma = 1, beta = 0; right-padded lengths drawn uniformly from an
integer range.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
import zlib
from dataclasses import dataclass
from typing import List, Optional

import numpy as np

_U64 = np.uint64
_GOLDEN = _U64(0x9E3779B97F4A7C15)
_M1 = _U64(0xBF58476D1CE4E5B9)
_M2 = _U64(0x94D049BB133111EB)


def _splitmix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser applied to ``z + golden`` (uint64, wrapping)."""
    with np.errstate(over="ignore"):
        z = z + _GOLDEN
        z = (z ^ (z >> _U64(30))) * _M1
        z = (z ^ (z >> _U64(27))) * _M2
    return z ^ (z >> _U64(31))


def stream_key(seed: int, name: str) -> int:
    """64-bit key of the named stream under ``seed``."""
    a = _splitmix64(np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))
    b = np.array([zlib.crc32(name.encode())], dtype=np.uint64)
    return int(_splitmix64(a ^ _splitmix64(b))[0])


def _normal_chunk(key: int, start: int, n: int) -> np.ndarray:
    idx = np.arange(start, start + n, dtype=np.uint64)
    k = np.uint64(key)
    with np.errstate(over="ignore"):
        ctr = idx * _U64(2) + k
    a = _splitmix64(ctr)
    with np.errstate(over="ignore"):
        b = _splitmix64(ctr + _U64(1))
    u1 = ((a >> _U64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)  # (0, 1)
    u2 = (b >> _U64(11)).astype(np.float64) * (2.0 ** -53)          # [0, 1)
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return z.astype(np.float32)


def normal(seed: int, name: str, n: int, start: int = 0, std: float = 1.0,
           threads: int = 0) -> np.ndarray:
    """``n`` float32 draws of N(0, std^2): elements [start, start+n) of a stream.

    The draw is made at unit variance in float64, rounded to float32, then
    multiplied by ``std`` in float32, so the same element is produced whatever
    the chunking.
    """
    key = stream_key(seed, name)
    chunk = 1 << 22
    if n <= chunk:
        out = _normal_chunk(key, start, n)
    else:
        out = np.empty(n, dtype=np.float32)
        starts = list(range(0, n, chunk))

        def work(s):
            out[s:s + min(chunk, n - s)] = _normal_chunk(key, start + s, min(chunk, n - s))

        nthr = threads or min(32, os.cpu_count() or 1)
        with _cf.ThreadPoolExecutor(nthr) as ex:
            list(ex.map(work, starts))
    if std != 1.0:
        out *= np.float32(std)
    return out


def uniform_int(seed: int, name: str, n: int, lo: int, hi: int) -> np.ndarray:
    """``n`` integers uniform on [lo, hi] (inclusive), int32."""
    key = stream_key(seed, name)
    idx = np.arange(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        r = _splitmix64(idx + np.uint64(key))
    span = np.uint64(hi - lo + 1)
    return (lo + (r % span).astype(np.int64)).astype(np.int32)


# --------------------------------------------------------------------------
# Workload table
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Shape:
    B: int
    S: int
    d_model: int
    n_heads: int
    d_ff: int
    n_layers: int
    causal: bool
    len_lo: Optional[int] = None   # None: every sequence is full length
    len_hi: Optional[int] = None
    name: str = ""

    @property
    def head_dim(self) -> int:
        return self.d_model // self.n_heads

    @property
    def tokens(self) -> int:
        return self.B * self.S


# The five benchmark shapes (the TechJam 2026 problem 3 shape matrix).
# Index 0 is the small latency-bound case.
WORKLOADS: List[Shape] = [
    Shape(1, 128, 128, 4, 512, 4, True, name="B1_S128_D128_causal"),
    Shape(64, 1024, 128, 4, 512, 4, True, 512, 1024, name="B64_S1024_D128_causal_ragged"),
    Shape(10000, 128, 128, 4, 512, 4, False, 32, 128, name="B10000_S128_D128_keymask_ragged"),
    Shape(16, 512, 1024, 4, 4096, 4, True, name="B16_S512_D1024_H4_causal"),
    Shape(32, 100000, 1024, 16, 4096, 1, True, name="B32_S100000_D1024_H16_causal"),
]


def lengths(seed: int, shape: Shape) -> np.ndarray:
    """Right-padded sequence lengths, int32 [B]."""
    if shape.len_lo is None:
        return np.full(shape.B, shape.S, dtype=np.int32)
    return uniform_int(seed, "lengths", shape.B, shape.len_lo, shape.len_hi)


def input_x(seed: int, shape: Shape, batches: Optional[np.ndarray] = None,
            threads: int = 0) -> np.ndarray:
    """x ~ N(0, 1) float32 [B, S, D] (or only the listed batch rows)."""
    row = shape.S * shape.d_model
    if batches is None:
        return normal(seed, "x", shape.B * row, threads=threads).reshape(shape.B, shape.S, shape.d_model)
    out = np.empty((len(batches), shape.S, shape.d_model), dtype=np.float32)
    for i, b in enumerate(batches):
        out[i] = normal(seed, "x", row, start=int(b) * row, threads=threads).reshape(shape.S, shape.d_model)
    return out


@dataclass
class LayerParams:
    wq: np.ndarray
    bq: np.ndarray
    wk: np.ndarray
    bk: np.ndarray
    wv: np.ndarray
    bv: np.ndarray
    wo: np.ndarray
    bo: np.ndarray
    ln1_g: np.ndarray
    ln1_b: np.ndarray
    ln2_g: np.ndarray
    ln2_b: np.ndarray
    w1: np.ndarray
    b1: np.ndarray
    w2: np.ndarray
    b2: np.ndarray

    FIELDS = ("wq", "bq", "wk", "bk", "wv", "bv", "wo", "bo", "ln1_g", "ln1_b",
              "ln2_g", "ln2_b", "w1", "b1", "w2", "b2")


@dataclass
class Params:
    layers: List[LayerParams]
    lnf_g: np.ndarray
    lnf_b: np.ndarray


def params(seed: int, shape: Shape, ln_affine: str = "identity",
           bias_std: float = 0.02) -> Params:
    """float32 parameters in nn.Linear layout ([out, in], row-major).

    ``ln_affine="identity"`` gives gamma = 1, beta = 0 (the benchmark recipe);
    ``"random"`` draws gamma ~ 1 + 0.1 N(0,1) and beta ~ 0.1 N(0,1), which the
    parity tests use so that a dropped or swapped affine term is visible.
    """
    D, F = shape.d_model, shape.d_ff

    def w(name, out_f, in_f):
        return normal(seed, name, out_f * in_f, std=float(1.0 / np.sqrt(in_f))).reshape(out_f, in_f)

    def b(name, n):
        return normal(seed, name, n, std=bias_std)

    def ln(name, n, base):
        if ln_affine == "identity":
            return np.full(n, base, dtype=np.float32)
        v = normal(seed, name, n, std=0.1)
        return (v + np.float32(base)).astype(np.float32)

    layers = []
    for l in range(shape.n_layers):
        p = f"l{l}."
        layers.append(LayerParams(
            wq=w(p + "wq", D, D), bq=b(p + "bq", D),
            wk=w(p + "wk", D, D), bk=b(p + "bk", D),
            wv=w(p + "wv", D, D), bv=b(p + "bv", D),
            wo=w(p + "wo", D, D), bo=b(p + "bo", D),
            ln1_g=ln(p + "ln1_g", D, 1.0), ln1_b=ln(p + "ln1_b", D, 0.0),
            ln2_g=ln(p + "ln2_g", D, 1.0), ln2_b=ln(p + "ln2_b", D, 0.0),
            w1=w(p + "w1", F, D), b1=b(p + "b1", F),
            w2=w(p + "w2", D, F), b2=b(p + "b2", D),
        ))
    return Params(layers=layers, lnf_g=ln("lnf_g", D, 1.0), lnf_b=ln("lnf_b", D, 0.0))
