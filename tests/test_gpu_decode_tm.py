"""GPU parity of the tensor-memory decode kernel (weights converted into
tensor memory as the 128-row A operand of tcgen05.mma, tokens as the B
operand, per-chunk group scales folded in by reduction warps; selected with
SPEAR_DECODE_TM=1) against the CPU oracle.

Source: SPEAR explainer, Technical Summary 2.1 A (y = W4 x + alpha g(x) B A x)
and 2.2 A (decode: compensator fused into the same launch)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from spear_testutil import (check_close, gpu_layer, make_layer, make_tokens, oracle_layer, sample_columns,
                            to_dev_u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _tensor_memory_kernel(monkeypatch):
    monkeypatch.setenv("SPEAR_DECODE_TM", "1")


def _run(layer, x_bits, out_dtype=1):
    from quantized_gemm_error_gb300 import spear
    y = spear.spear_linear_decode(layer, to_dev_u16(x_bits, torch.bfloat16), out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert spear.spear_get_device_status() == 0
    return y


# several row groups and chunks, ragged row groups, every token-tile width (16 / 32 / 64)
@pytest.mark.parametrize("N,K,G,sym,r,M", [
    (64, 128, 128, True, 16, 1),            # one chunk: the cluster shrinks to one CTA
    (192, 384, 128, False, 16, 3),
    (1024, 1024, 1024, True, 16, 16),       # per-channel: sums over the K slice in tensor memory
    (512, 2048, 128, False, 32, 9),
    (512, 1024, 128, False, 32, 24),
    (256, 2048, 2048, True, 64, 32),
    (320, 1152, 128, False, 64, 33),
    (256, 1024, 1024, False, 32, 64),
    (2048, 1024, 128, False, 32, 64),       # 64 tokens, one 128-row slice per row group: many row groups
    (1024, 1024, 128, True, 0, 5),          # rank 0: plain W4
])
def test_tm_decode_matches_oracle(N, K, G, sym, r, M):
    lay, rng = make_layer(N, K, r, seed=900 + N + M)
    x = make_tokens(rng, M, K, outlier_frac=0.01)
    L = gpu_layer(lay, G, sym)
    ref = oracle.linear(oracle_layer(lay, G, sym), x, nthreads=8)
    check_close(_run(L, x), ref)
    check_close(_run(L, x, out_dtype=0), ref)


@pytest.mark.parametrize("N,K,M", [(4096, 11008, 1), (11008, 4096, 16), (4096, 4096, 64)])
def test_tm_decode_llama7b_shapes_sampled(N, K, M):
    lay, rng = make_layer(N, K, 32, seed=17 + N + K + M)
    x = make_tokens(rng, M, K, outlier_frac=0.01)
    L = gpu_layer(lay, 128, False)
    cols = sample_columns(N, 192, seed=M)
    ref = oracle.linear(oracle_layer(lay, 128, False), x, n_idx=cols, nthreads=8)
    y = _run(L, x)
    check_close(y[:, torch.from_numpy(cols).cuda()], ref)


def test_tm_decode_very_wide_layer_twelve_tokens():
    """131072 x 128 at 12 tokens (one chunk: clusters of one CTA, many row groups)."""
    N, K, r = 131072, 128, 64
    lay, rng = make_layer(N, K, r, seed=24)
    x = make_tokens(rng, 12, K, outlier_frac=0.01)
    L = gpu_layer(lay, 128, False)
    cols = sample_columns(N, 256, seed=3)
    ref = oracle.linear(oracle_layer(lay, 128, False), x, n_idx=cols, nthreads=8)
    check_close(_run(L, x)[:, torch.from_numpy(cols).cuda()], ref)


def test_tm_gate_zero_and_comp_off_agree():
    """b_g = -1e4 drives the gate to 0: the output equals the compensator-off output bit for bit."""
    lay, rng = make_layer(512, 2048, 32, seed=31)
    x = make_tokens(rng, 7, 2048, outlier_frac=0.01)
    off = _run(gpu_layer(lay, 128, False, comp=False), x)
    zero = _run(gpu_layer(lay, 128, False, b_g=-1.0e4), x)
    assert torch.equal(off, zero)


@pytest.mark.parametrize("M", [1, 12, 40])
def test_tm_decode_vector_gate(M):
    from test_gpu_vector_gate import _layers
    L, OL, g, rng = _layers(512, 1024, 128, False, 32, 8, seed=400 + M)
    x = make_tokens(rng, M, 1024, outlier_frac=0.01)
    ref, _ = oracle.linear_vector_gate(OL, x, *g, nthreads=8)
    check_close(_run(L, x), ref)


def test_tm_decode_matches_default_kernel():
    """Same layer and tokens through the default kernels and this one: both
    within the tolerance of each other's reference, and close to each other."""
    lay, rng = make_layer(1024, 4096, 32, seed=5)
    x = make_tokens(rng, 4, 4096, outlier_frac=0.01)
    L = gpu_layer(lay, 128, False)
    y_tm = _run(L, x).cpu().numpy()
    import os
    os.environ["SPEAR_DECODE_TM"] = "0"
    try:
        y_def = _run(L, x).cpu().numpy()
    finally:
        os.environ["SPEAR_DECODE_TM"] = "1"
    rms = float(np.sqrt(np.mean(y_def.astype(np.float64) ** 2)))
    assert np.abs(y_tm - y_def).max() <= 1e-3 * rms
