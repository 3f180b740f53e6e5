"""Seeded synthetic inputs for the gated W4 + low-rank compensated linear layer.

This module only draws random numbers and casts them to the input dtypes; it
holds none of the method's arithmetic.  Both the CUDA path's tests/benchmark
and the oracle read their inputs from here, so the two always see the same
bytes.

Generator: numpy PCG64 (``numpy.random.default_rng(seed)``), standard normals
drawn in float32 and scaled.  Draw order per layer: W, A, B, w_g, x, outlier
channel set.  bf16 values are returned as uint16 bit patterns (round to
nearest even from float32).

Workloads follow the shapes and value distributions of Llama-style decoder
linears at 4-bit weight quantisation (the SPEAR explainer, Technical Summary
3.1, reports on Llama models from 1B to 70B; no dataset or trained weight is
used here -- every tensor is random).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = ["f32_to_bf16_bits", "bf16_bits_to_f32", "LayerInputs", "make_layer", "make_tokens",
           "WORKLOADS", "workload"]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Cast float32 -> bfloat16 (round to nearest even), returned as uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class LayerInputs:
    """One layer's raw inputs (before quantisation)."""
    N: int
    K: int
    r: int
    W: np.ndarray            # fp32 [N][K]
    A: np.ndarray            # bf16 bits [r][K]
    B: np.ndarray            # bf16 bits [N][r]
    w_g: np.ndarray          # bf16 bits [K]
    b_g: float = 0.0
    alpha: float = 1.0
    meta: dict = field(default_factory=dict)


def make_layer(N: int, K: int, r: int, seed: int = 0, *, w_std: float = 0.02,
               ab_std: float = 0.01, wg_std: float = 0.05, b_g: float = 0.0,
               alpha: float = 1.0) -> tuple[LayerInputs, np.random.Generator]:
    """W ~ N(0, w_std) fp32; A, B ~ N(0, ab_std) bf16; w_g ~ N(0, wg_std) bf16.

    Returns the layer and the generator, positioned for the token draws."""
    rng = np.random.default_rng(seed)
    W = rng.standard_normal((N, K), dtype=np.float32) * np.float32(w_std)
    A = f32_to_bf16_bits(rng.standard_normal((r, K), dtype=np.float32) * np.float32(ab_std))
    B = f32_to_bf16_bits(rng.standard_normal((N, r), dtype=np.float32) * np.float32(ab_std))
    w_g = f32_to_bf16_bits(rng.standard_normal((K,), dtype=np.float32) * np.float32(wg_std))
    return LayerInputs(N, K, r, W, A, B, w_g, b_g, alpha), rng


def make_tokens(rng: np.random.Generator, M: int, K: int, *, outlier_frac: float = 0.0,
                outlier_scale: float = 20.0) -> np.ndarray:
    """x ~ N(0, 1) [M][K]; a fixed seeded set of floor(outlier_frac*K) channels
    is multiplied by outlier_scale; returned as bf16 bits."""
    x = rng.standard_normal((M, K), dtype=np.float32)
    n_out = int(np.floor(outlier_frac * K))
    if n_out > 0:
        ch = rng.choice(K, size=n_out, replace=False)
        x[:, ch] *= np.float32(outlier_scale)
    return f32_to_bf16_bits(x)


# Named workloads: shape lists and quantisation formats of the synthetic
# Llama-shaped layers the library is tested and measured on.
WORKLOADS = {
    # single layer, per-output-channel symmetric int4, rank 16
    "layer1024_sym_r16": dict(shapes=[(1024, 1024)], G=None, sym=True, r=16,
                             decode_M=[1, 16], prefill_M=[], outlier_frac=0.0),
    # Llama-7B decoder linears (K, N): 4096x4096, 4096x11008, 11008x4096;
    # int4 group 128 asymmetric with uint4 zero points, rank 32
    "llama7b_decode_g128_r32": dict(shapes=[(4096, 4096), (4096, 11008), (11008, 4096)], G=128,
                                    sym=False, r=32, decode_M=[1, 4, 16, 64], prefill_M=[],
                                    outlier_frac=0.01),
    "llama7b_prefill_g128_r32": dict(shapes=[(4096, 4096), (4096, 11008), (11008, 4096)], G=128,
                                     sym=False, r=32, decode_M=[], prefill_M=[512, 2048, 8192],
                                     outlier_frac=0.01),
    # Llama-7B 32-block decoder stack: per block q, k, v, o (4096x4096), gate, up
    # (4096x11008), down (11008x4096); per-output-channel symmetric int4;
    # compensators (rank 64) on a layer mask of 4 of the 32 blocks, the other
    # blocks plain W4; one mixed step = a 1024-token prefill chunk plus 32
    # decode tokens (1056 tokens on the prefill path, 32 on the decode path)
    "llama7b_stack_sym_r64": dict(shapes=[(4096, 4096)] * 4 + [(4096, 11008)] * 2 + [(11008, 4096)],
                                  G=None, sym=True, r=64, blocks=32, masked_blocks=4,
                                  decode_M=[32], prefill_M=[1056], outlier_frac=0.0),
    # Llama-70B linears, group 128 asymmetric, rank 64
    "llama70b_g128_r64": dict(shapes=[(8192, 8192), (8192, 28672), (28672, 8192)], G=128, sym=False,
                              r=64, decode_M=[1, 8, 32], prefill_M=[256, 512, 1024, 2048, 4096],
                              outlier_frac=0.01),
}


def workload(name: str) -> dict:
    return dict(WORKLOADS[name])
