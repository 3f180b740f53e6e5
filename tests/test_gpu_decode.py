"""GPU parity for spear_linear_decode (one fused launch, M <= 64) against the
CPU oracle, on the workloads' shapes and value distributions.

Source: SPEAR explainer, Technical Summary 2.1 A (y = W4 x + alpha g(x) B A x)
and 2.2 A (decode: compensator fused into the GEMM epilogue)."""
import numpy as np
import pytest
import torch

import oracle
from spear_testutil import (check_close, gpu_layer, make_layer, make_tokens, oracle_layer, sample_columns,
                            to_dev_u16)

pytestmark = pytest.mark.gpu


def _spear():
    from quantized_gemm_error_gb300 import spear
    return spear


def _run(layer, x_bits, out_dtype=0, ws=None):
    sp = _spear()
    x = to_dev_u16(x_bits, torch.bfloat16)
    y = sp.spear_linear_decode(layer, x, out_dtype=out_dtype, workspace=ws)
    torch.cuda.synchronize()
    assert sp.spear_get_device_status() == 0
    return y


# small shapes the oracle finishes in seconds: several tiles, ragged token tiles
@pytest.mark.parametrize("N,K,G,sym,r,M", [
    (64, 128, 128, True, 16, 1),
    (192, 384, 128, False, 16, 3),
    (1024, 1024, 1024, True, 16, 1),        # 1024^2 per-channel symmetric, rank 16
    (1024, 1024, 1024, True, 16, 16),
    (512, 2048, 128, False, 32, 9),
    (512, 1024, 128, False, 32, 24),        # 17-32 tokens: tensor-core kernel, 32 token rows
    (256, 2048, 2048, True, 64, 32),
    (320, 1152, 128, False, 64, 33),
    (256, 1024, 1024, False, 32, 64),
    # tensor-core kernel, K units not a multiple of the cluster: units split
    # into halves between CTAs (11 units over clusters of 8, 9 over clusters
    # of 6: three split each), group and per-channel scales
    (512, 2816, 128, False, 32, 40),
    (512, 2304, 2304, True, 32, 64),
    (1024, 1024, 128, True, 0, 5),          # rank 0: plain W4
])
def test_decode_matches_oracle(N, K, G, sym, r, M):
    lay, rng = make_layer(N, K, r, seed=100 + N + M)
    x = make_tokens(rng, M, K, outlier_frac=0.01)
    L = gpu_layer(lay, G, sym)
    ref = oracle.linear(oracle_layer(lay, G, sym), x, nthreads=8)
    check_close(_run(L, x), ref)
    check_close(_run(L, x, out_dtype=1), ref)             # fp32 out: strict 1e-2 rms


@pytest.mark.parametrize("N,K,M", [(4096, 4096, 1), (11008, 4096, 4), (4096, 11008, 16), (4096, 4096, 64)])
def test_decode_llama7b_shapes_sampled(N, K, M):
    """Full Llama-7B shapes (int4 g128 asymmetric, rank 32, 1% outlier channels),
    checked on sampled output rows the oracle computes one by one."""
    lay, rng = make_layer(N, K, 32, seed=7 + N + K + M)
    x = make_tokens(rng, M, K, outlier_frac=0.01)
    L = gpu_layer(lay, 128, False)
    cols = sample_columns(N, 192, seed=M)
    ref = oracle.linear(oracle_layer(lay, 128, False), x, n_idx=cols, nthreads=8)
    y = _run(L, x)
    check_close(y[:, torch.from_numpy(cols).cuda()], ref)


def test_decode_very_wide_layer():
    """131072 output rows x 128.  One token runs (a warp-level block owns ~56
    16-row tiles, one block per SM).  At 12 tokens neither kernel can keep all
    its blocks resident (the warp-level plan outgrows shared memory; the
    tensor-core kernel would need 512 co-resident tile clusters), and the call
    says so instead of launching."""
    from quantized_gemm_error_gb300 import spear
    N, K, r = 131072, 128, 64
    lay, rng = make_layer(N, K, r, seed=24)
    L = gpu_layer(lay, 128, False)
    x = make_tokens(rng, 1, K, outlier_frac=0.01)
    ref = oracle.linear(oracle_layer(lay, 128, False), x, nthreads=8)
    check_close(_run(L, x), ref)
    with pytest.raises(spear.SpearError) as e:
        _run(L, make_tokens(rng, 12, K))
    assert spear.STATUS_NAMES[e.value.status] == "SPEAR_ERR_UNSUPPORTED"


def test_correction_term_alone():
    """Delta = y(comp on) - y(comp off) against the oracle's alpha g B (A x) (fp32 out)."""
    N, K, G, r, M = 1024, 2048, 128, 32, 7
    lay, rng = make_layer(N, K, r, seed=21)
    x = make_tokens(rng, M, K, outlier_frac=0.01)
    L = gpu_layer(lay, G, False)
    _, corr, _ = oracle.linear(oracle_layer(lay, G, False), x, nthreads=8, want_corr=True)
    d = _run(L, x, out_dtype=1) - _run(L.with_comp(False), x, out_dtype=1)
    check_close(d, corr, "correction")


def test_gate_zero_and_comp_off_are_bit_identical():
    N, K, r, M = 2048, 1024, 32, 5
    lay, rng = make_layer(N, K, r, seed=22)
    x = make_tokens(rng, M, K)
    L_on = gpu_layer(lay, 128, False, b_g=-1e30)           # sigmoid(-inf) = 0
    L_off = L_on.with_comp(False)
    assert torch.equal(_run(L_on, x, out_dtype=1), _run(L_off, x, out_dtype=1))
    assert torch.equal(_run(L_on, x), _run(L_off, x))


def test_workspace_is_reusable_across_calls_and_shapes():
    """The decode workspace's synchronisation words return to zero after every
    call, so one buffer serves a sequence of calls with different M and
    layers (same stream)."""
    sp = _spear()
    lays = []
    for i, (N, K) in enumerate([(1024, 1024), (512, 2048)]):
        lay, rng = make_layer(N, K, 32, seed=30 + i)
        lays.append((gpu_layer(lay, 128, False), rng, K))
    size = max(sp.spear_decode_workspace_bytes(L, M) for L, _, _ in lays for M in (1, 16, 64))
    ws = sp.new_workspace(size, "cuda")
    for M in (1, 16, 64, 3, 1):
        for L, rng, K in lays:
            x = make_tokens(rng, M, K)
            fresh = _run(L, x)
            again = _run(L, x, ws=ws)
            assert torch.equal(fresh, again)
    assert not ws[:16].any(), "workspace sync words not left zeroed"


def test_token_permutation_permutes_rows():
    N, K, r, M = 1024, 2048, 16, 12
    lay, rng = make_layer(N, K, r, seed=23)
    x = make_tokens(rng, M, K)
    L = gpu_layer(lay, 128, False)
    perm = np.random.default_rng(0).permutation(M)
    y = _run(L, x, out_dtype=1)
    yp = _run(L, x[perm], out_dtype=1)
    assert torch.equal(y[torch.from_numpy(perm).cuda()], yp)


def test_empty_batch_is_a_no_op():
    """M = 0 on both paths: nothing to read or write, SPEAR_OK, an empty y;
    M = 65 on the decode path is refused."""
    from quantized_gemm_error_gb300 import spear
    lay, rng = make_layer(512, 1024, 32, seed=25)
    L = gpu_layer(lay, 128, False)
    x0 = torch.empty(0, 1024, dtype=torch.bfloat16, device="cuda")
    assert spear.spear_decode_workspace_bytes(L, 0) == 0
    assert spear.spear_prefill_workspace_bytes(L, 0) == 0
    yd = spear.spear_linear_decode(L, x0)
    yp = spear.spear_linear_prefill(L, x0)
    torch.cuda.synchronize()
    assert yd.shape == (0, 512) and yp.shape == (0, 512)
    assert spear.spear_get_device_status() == 0
    with pytest.raises(spear.SpearError):
        spear.spear_linear_decode(L, to_dev_u16(make_tokens(rng, 65, 1024), torch.bfloat16))


def test_calls_without_a_workspace_reuse_one_per_stream():
    """Calls made without a workspace share the binding's one per (device,
    stream): made and zeroed once on the call's stream, reused after."""
    from quantized_gemm_error_gb300 import spear
    lay, rng = make_layer(512, 1024, 32, seed=77)
    L = gpu_layer(lay, 128, False)
    ref = oracle.linear(oracle_layer(lay, 128, False), make_tokens(np.random.default_rng(1), 3, 1024), nthreads=8)
    x = to_dev_u16(make_tokens(np.random.default_rng(1), 3, 1024), torch.bfloat16)
    spear.reset_default_workspaces()
    side = torch.cuda.Stream()
    outs = []
    for _ in range(3):
        with torch.cuda.stream(side):
            outs.append(spear.spear_linear_decode(L, x, out_dtype=spear.OUT_F32, stream=side))
    torch.cuda.synchronize()
    assert spear.spear_get_device_status() == 0
    assert len([k for k in spear._default_ws if k[0] == "decode"]) == 1
    for y in outs:
        check_close(y, ref)
    spear.reset_default_workspaces()
    assert not spear._default_ws


@pytest.mark.parametrize("N,K,G,sym,r,M", [
    (512, 2048, 128, False, 32, 3),          # tokens staged in fp16 (M <= 8)
    (1024, 1024, 1024, True, 16, 8),         # staged, per-channel scales
    (512, 2048, 128, False, 32, 12),         # bf16 tokens from L1
    (512, 1024, 128, False, 32, 24),         # tensor-core kernel, fp16 token tiles
    (256, 1024, 1024, False, 32, 64),
    (512, 2048, 2048, True, 32, 40),         # tensor-core kernel, per-channel scales (the scale after the sum)
    (512, 2816, 128, False, 32, 40),         # tensor-core kernel with split K units (fp32 rows over half units)
])
def test_decode_activations_of_any_magnitude(N, K, G, sym, r, M):
    """Tokens with |x| up to ~1e6 (beyond fp16): the fp16 launches scale each
    such token by a power of two and match the oracle."""
    from quantized_gemm_error_gb300.inputs import f32_to_bf16_bits
    from spear_testutil import bf16_bits_to_f32
    lay, rng = make_layer(N, K, r, seed=300 + N + M)
    x = bf16_bits_to_f32(make_tokens(rng, M, K, outlier_frac=0.01)).reshape(M, K)
    row_scale = np.ones(M, np.float32)
    row_scale[0::3] = 3.0e4                                  # max |x| ~ 1e6 with the x20 outliers
    x = x * row_scale[:, None]
    x[min(1, M - 1), 5] = 9.5e5                              # one huge value in an ordinary token
    x = f32_to_bf16_bits(x)
    L = gpu_layer(lay, G, sym)
    ref = oracle.linear(oracle_layer(lay, G, sym), x, nthreads=8)
    check_close(_run(L, x, out_dtype=1), ref)


@pytest.mark.parametrize("M", [3, 40])
def test_decode_reports_non_finite_activations(M):
    """A bf16 inf among the tokens is reported as SPEAR_ERR_INVALID_ARG on the
    launches that carry the tokens in fp16 (staged tokens, the tensor-core
    kernel); the output of that token is not defined."""
    from quantized_gemm_error_gb300 import spear
    lay, rng = make_layer(512, 2048, 32, seed=48 + M)
    x = make_tokens(rng, M, 2048, outlier_frac=0.01)
    x[min(1, M - 1), 300] = 0x7F80                          # bf16 +inf
    L = gpu_layer(lay, 128, False)
    spear.spear_linear_decode(L, to_dev_u16(x, torch.bfloat16), out_dtype=1)
    torch.cuda.synchronize()
    assert spear.STATUS_NAMES[spear.spear_get_device_status()] == "SPEAR_ERR_INVALID_ARG"
    assert spear.spear_get_device_status() == 0
