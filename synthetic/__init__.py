"""Seeded synthetic inputs for the W4A4 + LoRA linear layer.

This module only draws random numbers; it holds none of the method's
arithmetic (no quantisation, no packing, no matrix products).  Both the CUDA
path (through tests and ``bench.py``) and the CPU oracle are fed from here, so
that each side sees bit-identical inputs.

Distributions follow the workloads described on the pages:

* activations ``X`` ~ N(0, 1), with 1% of the input channels scaled by 20
  (outlier channels, as in the voice-model profile of the L4 blog post,
  section 2.1 "INT4 is too coarse"), stored as fp16;
* weights ``W`` ~ N(0, 0.02) in fp32 (the packer quantises them);
* LoRA factors ``L_down`` [K, r] and ``L_up`` [r, N] ~ N(0, 0.02), fp16
  (the rank-r low-rank branch of "2.1 ... needs LoRA correction");
* per-column affine ``colscale`` ~ U(0.5, 1.5) and ``bias`` ~ N(0, 0.1), fp16
  (the column-wise affine of the Blackwell W4A4 article, section 1).

Draw order is fixed: X, outlier channel indices, W, L_down, L_up, colscale,
bias.  Each call uses ``numpy.random.default_rng(seed)``.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

GROUP = 64  # quantisation group along K


@dataclass
class LinearCase:
    M: int
    K: int
    N: int
    r: int
    X: np.ndarray         # uint16 [M, K]  (fp16 bit patterns)
    W: np.ndarray         # float32 [N, K]
    L_down: np.ndarray    # uint16 [K, r]  (fp16 bits)
    L_up: np.ndarray      # uint16 [r, N]  (fp16 bits)
    colscale: np.ndarray  # uint16 [N]     (fp16 bits)
    bias: np.ndarray      # uint16 [N]     (fp16 bits)
    outliers: np.ndarray  # int64 [n_out] outlier channel indices


def _f16_bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a.astype(np.float16)).view(np.uint16)


def n_outlier_channels(K: int) -> int:
    """1% of the K input channels, rounded to nearest (10 at K=1024)."""
    return int(round(0.01 * K))


def make_activations(rng: np.random.Generator, M: int, K: int):
    X = rng.standard_normal((M, K), dtype=np.float32)
    n_out = n_outlier_channels(K)
    idx = np.sort(rng.choice(K, size=n_out, replace=False)) if n_out > 0 else np.zeros(0, np.int64)
    if n_out:
        X[:, idx] *= np.float32(20.0)
    return _f16_bits(X), idx.astype(np.int64)


def make_linear_case(M: int, K: int, N: int, r: int = 32, seed=0) -> LinearCase:
    """One W4A4 linear layer's inputs, drawn in the fixed order above."""
    rng = np.random.default_rng(seed)
    X, idx = make_activations(rng, M, K)
    W = (rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)).astype(np.float32)
    L_down = _f16_bits(rng.standard_normal((K, r), dtype=np.float32) * np.float32(0.02))
    L_up = _f16_bits(rng.standard_normal((r, N), dtype=np.float32) * np.float32(0.02))
    colscale = _f16_bits(rng.uniform(0.5, 1.5, size=N).astype(np.float32))
    bias = _f16_bits(rng.standard_normal(N, dtype=np.float32) * np.float32(0.1))
    return LinearCase(M, K, N, r, X, np.ascontiguousarray(W), L_down, L_up, colscale, bias, idx)


# Shapes of the workloads (sizes only).
SINGLE_LINEAR = dict(M=64, K=1024, N=1024, r=32)
DECODER_LAYER_M700 = {
    "qkv": dict(M=700, K=1024, N=4096, r=32),
    "o": dict(M=700, K=2048, N=1024, r=32),
    "gate_up": dict(M=700, K=1024, N=6144, r=32),
    "down": dict(M=700, K=3072, N=1024, r=32),
}
SMALL_M_SWEEP = [dict(M=m, K=4096, N=4096, r=32) for m in (1, 4, 16, 32, 76)]
PREFILL = {
    "gate_up_style": dict(M=8192, K=4096, N=14336, r=32),
    "down_style": dict(M=8192, K=14336, N=4096, r=32),
}


def random_codes(rng: np.random.Generator, shape, lo=-8, hi=7) -> np.ndarray:
    """Uniform integer codes in [lo, hi] (edge-case tests: the full INT4 range)."""
    return rng.integers(lo, hi + 1, size=shape, dtype=np.int64).astype(np.int8)


def random_f16(rng: np.random.Generator, shape, lo: float, hi: float) -> np.ndarray:
    return _f16_bits(rng.uniform(lo, hi, size=shape).astype(np.float32))


# ---- config 5: a stack of decoder layers -------------------------------------
# Each layer has the four linears below, in this order; every linear of every
# layer gets fresh weights from ``default_rng([0, layer, j])`` (j = position in
# the layer), drawn in the order W, L_down, L_up, colscale, bias.  The stack's
# input is ``make_activations`` of ``default_rng(seed)`` at K = 1024.
STACK_LAYERS = 28
STACK_LINEARS = (("qkv", 1024, 4096), ("o", 2048, 1024), ("gate_up", 1024, 6144), ("down", 3072, 1024))


@dataclass
class StackLinear:
    layer: int
    j: int
    name: str
    K: int
    N: int
    r: int
    W: np.ndarray         # float32 [N, K]
    L_down: np.ndarray    # uint16 [K, r]
    L_up: np.ndarray      # uint16 [r, N]
    colscale: np.ndarray  # uint16 [N]
    bias: np.ndarray      # uint16 [N]


def make_stack_linear(layer: int, j: int, r: int = 32) -> StackLinear:
    name, K, N = STACK_LINEARS[j]
    rng = np.random.default_rng([0, layer, j])
    W = (rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)).astype(np.float32)
    L_down = _f16_bits(rng.standard_normal((K, r), dtype=np.float32) * np.float32(0.02))
    L_up = _f16_bits(rng.standard_normal((r, N), dtype=np.float32) * np.float32(0.02))
    colscale = _f16_bits(rng.uniform(0.5, 1.5, size=N).astype(np.float32))
    bias = _f16_bits(rng.standard_normal(N, dtype=np.float32) * np.float32(0.1))
    return StackLinear(layer, j, name, K, N, r, np.ascontiguousarray(W), L_down, L_up, colscale, bias)


def make_stack_input(M: int, seed: int = 0) -> np.ndarray:
    """The stack's first input, fp16 bits uint16 [M, 1024]."""
    X, _ = make_activations(np.random.default_rng(seed), M, STACK_LINEARS[0][1])
    return X


def stack_next_k(j: int) -> int:
    """Columns of linear j's output that feed the next linear (wrapping to the next layer)."""
    return STACK_LINEARS[(j + 1) % len(STACK_LINEARS)][1]
