"""The give-up path of a bounded device wait, made to run out on purpose by
the host (no GPU fault, no trap): the decode kernels' streamer blocks (warp-
level kernel) and tile CTAs (tensor-core kernel) wait for the T that their
producers publish through the workspace.

A decode workspace starts with the producers' arrival counter (the last
producer to arrive publishes T).  Presetting that counter far past the
producer count means no producer is ever the last, so T is never published
and every wait for it runs out.  With a 1 ms limit
(spear_set_wait_limit_ns) the call must return, report SPEAR_ERR_TIMEOUT
through spear_get_device_status, and have left the compensator term out; after
spear_workspace_init the same workspace serves a correct call again.

Source: SPEAR explainer, Technical Summary 2.2 A (the decode kernel, one
launch per layer); the bounded waits are this library's."""
import numpy as np
import pytest
import torch

import oracle
from spear_testutil import check_close, gpu_layer, make_layer, make_tokens, oracle_layer, to_dev_u16

pytestmark = pytest.mark.gpu


def test_decode_wait_runs_out_then_workspace_recovers():
    from quantized_gemm_error_gb300 import spear
    N, K, G, sym, r, M = 1024, 2048, 128, False, 32, 4      # warp-level kernel with producer blocks
    lay, rng = make_layer(N, K, r, seed=61)
    x_bits = make_tokens(rng, M, K, outlier_frac=0.01)
    x = to_dev_u16(x_bits, torch.bfloat16)
    L = gpu_layer(lay, G, sym)
    ref = oracle.linear(oracle_layer(lay, G, sym), x_bits, nthreads=8)
    ws = spear.new_workspace(spear.spear_decode_workspace_bytes(L, M), "cuda")

    y = spear.spear_linear_decode(L, x, out_dtype=spear.OUT_F32, workspace=ws)
    torch.cuda.synchronize()
    assert spear.spear_get_device_status() == 0
    check_close(y, ref)

    # no producer will be the last to arrive: T is never published
    ws.view(torch.int32)[0] = 1 << 30
    spear.spear_set_wait_limit_ns(1_000_000)
    try:
        y_timed_out = spear.spear_linear_decode(L, x, out_dtype=spear.OUT_F32, workspace=ws)
        torch.cuda.synchronize()                              # the call returned and the launch finished
        assert spear.STATUS_NAMES[spear.spear_get_device_status()] == "SPEAR_ERR_TIMEOUT"
        assert spear.spear_get_device_status() == 0           # read and cleared
    finally:
        spear.spear_set_wait_limit_ns(0)

    # the blocks that gave up left alpha g B T out: the plain W4 output, bit for bit
    y_plain = spear.spear_linear_decode(L.with_comp(False), x, out_dtype=spear.OUT_F32)
    torch.cuda.synchronize()
    assert spear.spear_get_device_status() == 0
    assert torch.equal(y_timed_out, y_plain)

    # zeroed again, the same workspace serves a correct call
    spear.spear_workspace_init(ws)
    y_again = spear.spear_linear_decode(L, x, out_dtype=spear.OUT_F32, workspace=ws)
    torch.cuda.synchronize()
    assert spear.spear_get_device_status() == 0
    check_close(y_again, ref)


def test_tensor_core_decode_wait_runs_out_then_workspace_recovers():
    """The tensor-core kernel (40 tokens): its producer clusters count their
    published row tiles in the workspace's first word and the last one forms
    T; preset past the cluster count, T is never published, every tile CTA's
    wait runs out and the compensator term is left out."""
    from quantized_gemm_error_gb300 import spear
    N, K, G, sym, r, M = 512, 2048, 128, False, 32, 40
    lay, rng = make_layer(N, K, r, seed=63)
    x_bits = make_tokens(rng, M, K, outlier_frac=0.01)
    x = to_dev_u16(x_bits, torch.bfloat16)
    L = gpu_layer(lay, G, sym)
    ref = oracle.linear(oracle_layer(lay, G, sym), x_bits, nthreads=8)
    ws = spear.new_workspace(spear.spear_decode_workspace_bytes(L, M), "cuda")

    y = spear.spear_linear_decode(L, x, out_dtype=spear.OUT_F32, workspace=ws)
    torch.cuda.synchronize()
    assert spear.spear_get_device_status() == 0
    check_close(y, ref)

    ws.view(torch.int32)[0] = 1 << 30
    spear.spear_set_wait_limit_ns(1_000_000)
    try:
        y_timed_out = spear.spear_linear_decode(L, x, out_dtype=spear.OUT_F32, workspace=ws)
        torch.cuda.synchronize()
        assert spear.STATUS_NAMES[spear.spear_get_device_status()] == "SPEAR_ERR_TIMEOUT"
        assert spear.spear_get_device_status() == 0
    finally:
        spear.spear_set_wait_limit_ns(0)

    y_plain = spear.spear_linear_decode(L.with_comp(False), x, out_dtype=spear.OUT_F32)
    torch.cuda.synchronize()
    assert spear.spear_get_device_status() == 0
    assert torch.equal(y_timed_out, y_plain)

    spear.spear_workspace_init(ws)
    y_again = spear.spear_linear_decode(L, x, out_dtype=spear.OUT_F32, workspace=ws)
    torch.cuda.synchronize()
    assert spear.spear_get_device_status() == 0
    check_close(y_again, ref)


def test_wait_limit_setting_leaves_correct_calls_correct():
    """A limit far above the legitimate wait changes nothing; 0 restores the default."""
    from quantized_gemm_error_gb300 import spear
    lay, rng = make_layer(512, 1024, 32, seed=62)
    x_bits = make_tokens(rng, 9, 1024, outlier_frac=0.01)
    L = gpu_layer(lay, 128, False)
    ref = oracle.linear(oracle_layer(lay, 128, False), x_bits, nthreads=8)
    for limit in (10 ** 9, 0):
        spear.spear_set_wait_limit_ns(limit)
        y = spear.spear_linear_decode(L, to_dev_u16(x_bits, torch.bfloat16), out_dtype=spear.OUT_F32)
        torch.cuda.synchronize()
        assert spear.spear_get_device_status() == 0
        check_close(y, ref)
    assert np.isfinite(ref).all()
