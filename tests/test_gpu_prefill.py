"""GPU parity for spear_linear_prefill (tcgen05 tensor-core GEMM over int4
tiles, compensator fused into the K loop or run on a second stream) against
the CPU oracle.

Source: SPEAR explainer, Technical Summary 2.1 A (the layer) and 2.2 A
(prefill: compensator as a separate kernel overlapped with the GEMM)."""
import numpy as np
import pytest
import torch

import oracle
from quantized_gemm_error_gb300.inputs import f32_to_bf16_bits
from spear_testutil import (bf16_bits_to_f32, check_close, gpu_layer, make_layer, make_tokens, oracle_layer,
                            sample_columns, to_dev_u16)

pytestmark = pytest.mark.gpu

FUSED, STREAM = 1, 2


def _run(layer, x_bits, mode=FUSED, out_dtype=0):
    from quantized_gemm_error_gb300 import spear
    x = to_dev_u16(x_bits, torch.bfloat16)
    aux = torch.cuda.Stream()
    y = spear.spear_linear_prefill(layer, x, out_dtype=out_dtype, mode=mode, stream_aux=aux)
    torch.cuda.synchronize()
    assert spear.spear_get_device_status() == 0
    return y


@pytest.mark.parametrize("G,sym", [(128, True), (256, False)])
def test_prefill_single_tile_plain(G, sym):
    """One 128 x 256 tile, no compensator: per-channel (G = K) and grouped scales."""
    K = 256
    lay, rng = make_layer(256, K, 0, seed=40)
    x = make_tokens(rng, 128, K)
    g = K if G == 256 else G
    L = gpu_layer(lay, g, sym)
    ref = oracle.linear(oracle_layer(lay, g, sym), x, nthreads=8)
    check_close(_run(L, x, out_dtype=1), ref)


@pytest.mark.parametrize("N,K,G,sym,r,M", [
    (256, 256, 128, False, 0, 200),
    (512, 1024, 1024, True, 16, 130),
    (768, 1024, 128, False, 32, 300),
    (320, 2048, 128, False, 64, 257),       # ragged N tile (320 = 256 + 64) and ragged M
    (1024, 1024, 1024, True, 32, 512),
    (512, 1024, 128, False, 32, 1100),
    # 256-token tiles (10 column tiles, M ~ 2000: one wave of 256-token tiles
    # against two of 128-token ones on 152 SMs): ragged last tile, rank 16 /
    # 32 / 64 (64- and 128-byte T rows)
    (2560, 512, 128, False, 32, 2000),
    (2560, 512, 128, False, 64, 1950),
    (2560, 512, 128, True, 16, 2048),
    (2560, 512, 512, False, 0, 2000),       # per-channel scales, no compensator: 256-token tiles
    (2560, 512, 512, False, 32, 2000),      # per-channel scales with the compensator: 128-token tiles
])
@pytest.mark.parametrize("mode", [FUSED, STREAM])
def test_prefill_matches_oracle(N, K, G, sym, r, M, mode):
    lay, rng = make_layer(N, K, r, seed=41 + N + M + r)
    x = make_tokens(rng, M, K, outlier_frac=0.01)
    L = gpu_layer(lay, G, sym)
    ref = oracle.linear(oracle_layer(lay, G, sym), x, nthreads=8)
    check_close(_run(L, x, mode), ref)
    check_close(_run(L, x, mode, out_dtype=1), ref)


@pytest.mark.parametrize("mode", [FUSED, STREAM])
def test_prefill_correction_term_alone(mode):
    N, K, r, M = 512, 2048, 32, 160
    lay, rng = make_layer(N, K, r, seed=43)
    x = make_tokens(rng, M, K, outlier_frac=0.01)
    L = gpu_layer(lay, 128, False)
    _, corr, _ = oracle.linear(oracle_layer(lay, 128, False), x, nthreads=8, want_corr=True)
    d = _run(L, x, mode, out_dtype=1) - _run(L.with_comp(False), x, mode, out_dtype=1)
    check_close(d, corr, "correction")


@pytest.mark.parametrize("N,K,M", [(4096, 4096, 512), (11008, 4096, 2048), (4096, 11008, 512)])
def test_prefill_llama7b_shapes_sampled(N, K, M):
    lay, rng = make_layer(N, K, 32, seed=44 + N + K)
    x = make_tokens(rng, M, K, outlier_frac=0.01)
    L = gpu_layer(lay, 128, False)
    cols = sample_columns(N, 96, seed=1)
    ref = oracle.linear(oracle_layer(lay, 128, False), x, n_idx=cols, nthreads=8)
    idx = torch.from_numpy(cols).cuda()
    for mode in (FUSED, STREAM):
        check_close(_run(L, x, mode)[:, idx], ref)


@pytest.mark.parametrize("M", [16, 64])
def test_decode_and_prefill_agree(M):
    from quantized_gemm_error_gb300 import spear
    N, K, r = 1024, 2048, 32
    lay, rng = make_layer(N, K, r, seed=45)
    x_bits = make_tokens(rng, M, K, outlier_frac=0.01)
    L = gpu_layer(lay, 128, False)
    ref = oracle.linear(oracle_layer(lay, 128, False), x_bits, nthreads=8)
    yp = _run(L, x_bits, FUSED, out_dtype=1)
    yd = spear.spear_linear_decode(L, to_dev_u16(x_bits, torch.bfloat16), out_dtype=1)
    torch.cuda.synchronize()
    check_close(yp, ref)
    check_close(yd, ref)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert (yp - yd).abs().max().item() <= 2e-2 * rms


@pytest.mark.parametrize("N,K,M", [(512, 1024, 200), (2560, 512, 2000)])
def test_prefill_gate_zero_equals_plain(N, K, M):
    r = 32
    lay, rng = make_layer(N, K, r, seed=46)
    x = make_tokens(rng, M, K)
    L_on = gpu_layer(lay, 128, False, b_g=-1e30)
    y_on = _run(L_on, x, FUSED, 1)
    y_off = _run(L_on.with_comp(False), x, FUSED, 1)
    # the fused correction adds exact zeros (its own accumulator for 128-token
    # tiles, the main one for 256-token tiles)
    assert torch.equal(y_on, y_off)


def _huge_tokens(rng, M, K):
    """x ~ N(0, 1) with 1 % outlier channels x20, then rows scaled so some
    tokens reach |x| ~ 1e6 (beyond fp16), some stay ordinary, one mixes a huge
    and tiny values."""
    x = bf16_bits_to_f32(make_tokens(rng, M, K, outlier_frac=0.01)).reshape(M, K)
    row_scale = np.ones(M, np.float32)
    row_scale[0::3] = 3.0e4                                  # max |x| ~ 1e6 with the x20 outliers
    row_scale[1::7] = 1.5e3                                  # max ~ 1e5
    x = x * row_scale[:, None]
    x[2, 5] = 9.5e5                                          # one huge value in an ordinary token
    return f32_to_bf16_bits(x)


@pytest.mark.parametrize("N,K,G,sym,r,M,mode", [
    (256, 256, 128, False, 0, 200, FUSED),                   # no compensator: the row-wise fp16 copy
    (768, 1024, 128, False, 32, 300, FUSED),                 # 128-token tiles, correction in its own accumulator
    (768, 1024, 128, False, 32, 300, STREAM),                # concurrent stream: the up-projection adds unscaled
    (2560, 512, 128, False, 32, 2000, FUSED),                # 256-token tiles: the correction joins scaled accumulators
    (1024, 1024, 1024, True, 32, 512, FUSED),                # per-channel scales, K split
])
def test_prefill_activations_of_any_magnitude(N, K, G, sym, r, M, mode):
    """Tokens with |x| up to ~1e6 (beyond fp16) run on the fp16 GEMM through
    power-of-two token scaling and match the oracle."""
    lay, rng = make_layer(N, K, r, seed=47 + N + M)
    x = _huge_tokens(rng, M, K)
    L = gpu_layer(lay, G, sym)
    ref = oracle.linear(oracle_layer(lay, G, sym), x, nthreads=8)
    check_close(_run(L, x, mode, 1), ref)


def test_prefill_reports_non_finite_activations():
    from quantized_gemm_error_gb300 import spear
    lay, rng = make_layer(256, 256, 0, seed=47)
    x = make_tokens(rng, 128, 256)
    x[3, 7] = 0x7F80                                        # bf16 +inf
    L = gpu_layer(lay, 128, False)
    spear.spear_linear_prefill(L, to_dev_u16(x, torch.bfloat16), out_dtype=1)
    torch.cuda.synchronize()
    assert spear.spear_get_device_status() == 1
    assert spear.spear_get_device_status() == 0
