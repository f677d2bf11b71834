"""Seeded synthetic inputs for the quantized multi-row matmul.

This module is shared by the oracle-side tests and the GPU-side tests/bench;
it holds none of the method's arithmetic (no packing, no dequantization, no
dot products). It only draws random numbers and rounds them to the storage
formats the operation consumes:

* packed codes: independent uniform random uint32 words. Every bit of the
  LSB-first code stream is an independent fair coin, so every code of every
  width (4/5/6/8 bits, including codes that straddle two words) is uniform on
  [0, 2**bits) -- the distribution the workloads ask for -- without this module
  knowing the packing rule.
* scales: U[0.002, 0.02] drawn in float64, rounded to IEEE binary16 (RNE).
* biases: -2**(bits-1) * scale + N(0, 1e-3) (1e-3 is the standard deviation),
  computed in float64 from the already-rounded binary16 scale, then rounded to
  binary16 (RNE).
* activations x: N(0, 1) drawn in float64, rounded to binary32 (RNE) and then
  to bfloat16 (RNE).

Generator: numpy's PCG64 seeded per workload. Storage dtypes are returned as
raw bit patterns (uint16 for binary16 / bfloat16, uint32 for code words).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# Seed base for the named workloads: seed = SEED_BASE + workload index.
SEED_BASE = 0x51ED0000


def f64_to_f16_bits(v: np.ndarray) -> np.ndarray:
    """Round float64 to IEEE binary16 (numpy's RNE cast) and return raw bits."""
    return np.asarray(v, dtype=np.float64).astype(np.float16).view(np.uint16)


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round float64 -> binary32 (RNE) -> bfloat16 (RNE, ties to even) bits."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


@dataclass
class QmmInputs:
    x: np.ndarray        # uint16 [M, K]   bfloat16 bits
    words: np.ndarray    # uint32 [B, N, K*bits/32] packed code words
    scales: np.ndarray   # uint16 [B, N, K/group] binary16 bits
    biases: np.ndarray   # uint16 [B, N, K/group] binary16 bits
    M: int
    K: int
    N: int
    bits: int
    group: int
    banks: int


def gen_qmm(seed: int, M: int, K: int, N: int, bits: int, group: int, banks: int = 1,
            x_scale: float = 1.0) -> QmmInputs:
    """Synthetic inputs with the workloads' value distributions.

    ``banks`` independent weight sets (packed words, scales, biases) share one
    x. ``x_scale`` multiplies the N(0,1) activations before rounding (1.0 for
    every named workload).
    """
    if K % group or (K * bits) % 32:
        raise ValueError("K must be a multiple of group and K*bits of 32")
    rng = np.random.Generator(np.random.PCG64(seed))
    G = K // group
    wpr = K * bits // 32
    x = f64_to_bf16_bits(rng.standard_normal((M, K)) * x_scale)
    words = rng.integers(0, 1 << 32, size=(banks, N, wpr), dtype=np.uint64).astype(np.uint32)
    s = f64_to_f16_bits(rng.uniform(0.002, 0.02, size=(banks, N, G)))
    s_val = s.view(np.float16).astype(np.float64)
    b = f64_to_f16_bits(-float(1 << (bits - 1)) * s_val + rng.normal(0.0, 1e-3, size=(banks, N, G)))
    return QmmInputs(x=x, words=words, scales=s, biases=b, M=M, K=K, N=N, bits=bits,
                     group=group, banks=banks)


def gen_x(seed: int, M: int, K: int, x_scale: float = 1.0) -> np.ndarray:
    """Only the bfloat16 activations (same recipe as gen_qmm)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return f64_to_bf16_bits(rng.standard_normal((M, K)) * x_scale)


# The named workloads (shapes and formats of the pages' projections).
WORKLOADS = {
    # name: dict(M list, K, N, bits list, group, out, splits list, banks)
    "pr1_ref": dict(Ms=[1], K=2048, N=2048, bits=[4], group=64, out="f32", splits=[1], banks=1),
    "mlp_up": dict(Ms=[1, 2, 4, 8, 16], K=5120, N=17408, bits=[4], group=32, out="bf16",
                   splits=[1], banks=1),
    "down_longk": dict(Ms=[1, 8, 16], K=17408, N=5120, bits=[4], group=64, out="bf16",
                       splits=[1, 2, 4, 8], banks=1),
    "mixed_widths": dict(Ms=[8], K=5120, N=6144, bits=[5, 6, 8], group=32, out="bf16",
                         splits=[1], banks=1),
    "banked": dict(Ms=[1, 16], K=2048, N=8192, bits=[4], group=64, out="bf16", splits=[1],
                   banks=36),
    # lm_head-class projection: 8-bit codes over a ~152k vocabulary (661 MB of
    # codes, scales and biases streamed per call)
    "lm_head": dict(Ms=[1, 8, 16], K=4096, N=151936, bits=[8], group=64, out="bf16", splits=[1],
                    banks=1),
}
WORKLOAD_INDEX = {name: i for i, name in enumerate(WORKLOADS)}


def workload_seed(name: str) -> int:
    return SEED_BASE + WORKLOAD_INDEX[name]
