"""GPU parity for spear_linear_prefill (tcgen05 tensor-core GEMM over int4
tiles, compensator fused into the K loop or run on a second stream) against
the CPU oracle.

Source: SPEAR explainer, Technical Summary 2.1 A (the layer) and 2.2 A
(prefill: compensator as a separate kernel overlapped with the GEMM)."""
import numpy as np
import pytest
import torch

import oracle
from spear_testutil import check_close, gpu_layer, make_layer, make_tokens, oracle_layer, sample_columns, to_dev_u16

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


def test_prefill_reports_activations_beyond_fp16_range():
    from quantized_gemm_error_gb300 import spear
    lay, rng = make_layer(256, 256, 0, seed=47)
    x = make_tokens(rng, 128, 256)
    x[3, 7] = 0x4780                                        # bf16 65536: beyond the fp16 range
    L = gpu_layer(lay, 128, False)
    spear.spear_linear_prefill(L, to_dev_u16(x, torch.bfloat16), out_dtype=1)
    torch.cuda.synchronize()
    assert spear.spear_get_device_status() == 1
    assert spear.spear_get_device_status() == 0
