"""GPU parity at the full sizes of the remaining workloads, checked on sampled
output rows the oracle computes one by one:

* Llama-70B linears (8192x8192, 8192x28672, 28672x8192; int4 group 128
  asymmetric, rank 64, 1 % outlier channels x20): decode M in {1, 8, 32},
  prefill M in {256, 512, 1024, 2048, 4096};
* the Llama-7B prefill linears at their largest chunk, M = 8192;
* the Llama-7B decoder-block stack's layer shapes (per-output-channel symmetric
  int4; rank 64 on the masked blocks, plain W4 on the rest) at one mixed step:
  prefill M = 1056 (a 1024-token chunk and 32 decode tokens), decode M = 32.

Source: SPEAR explainer, Technical Summary 2.1 A (the layer) and 2.2 A (the
decode and prefill kernels)."""
import numpy as np
import pytest
import torch

import oracle
from quantized_gemm_error_gb300.inputs import workload
from spear_testutil import check_close, gpu_layer, make_layer, make_tokens, oracle_layer, sample_columns, to_dev_u16

pytestmark = pytest.mark.gpu

W70 = workload("llama70b_g128_r64")
STACK = workload("llama7b_stack_sym_r64")
P7 = workload("llama7b_prefill_g128_r32")

_held = {}


def _layer(N, K, r, G, sym, seed):
    """One full-size layer at a time (GPU copy and oracle form), reused by the
    consecutive cases of the same shape."""
    key = (N, K, r, G, sym, seed)
    if key not in _held:
        _held.clear()
        torch.cuda.empty_cache()
        lay, _ = make_layer(N, K, r, seed=seed)
        _held[key] = (gpu_layer(lay, G, sym), oracle_layer(lay, G, sym))
    return _held[key]


def _check(L, OL, M, K, N, phase, ncols, seed, outlier_frac):
    from quantized_gemm_error_gb300 import spear
    x = make_tokens(np.random.default_rng(seed), M, K, outlier_frac=outlier_frac)
    cols = sample_columns(N, ncols, seed=seed)
    ref = oracle.linear(OL, x, n_idx=cols, nthreads=8)
    xd = to_dev_u16(x, torch.bfloat16)
    y = spear.spear_linear_decode(L, xd) if phase == "decode" else spear.spear_linear_prefill(L, xd)
    torch.cuda.synchronize()
    assert spear.spear_get_device_status() == 0
    check_close(y[:, torch.from_numpy(cols).cuda()], ref)


@pytest.mark.parametrize("K,N,M", [(K, N, M) for (K, N) in W70["shapes"] for M in W70["decode_M"]])
def test_llama70b_decode_sampled(K, N, M):
    L, OL = _layer(N, K, W70["r"], W70["G"], W70["sym"], seed=N + K)
    _check(L, OL, M, K, N, "decode", 128, M, W70["outlier_frac"])


@pytest.mark.parametrize("K,N,M", [(K, N, M) for (K, N) in W70["shapes"] for M in W70["prefill_M"]])
def test_llama70b_prefill_sampled(K, N, M):
    L, OL = _layer(N, K, W70["r"], W70["G"], W70["sym"], seed=N + K)
    _check(L, OL, M, K, N, "prefill", 48 if M > 1024 else 96, M, W70["outlier_frac"])


@pytest.mark.parametrize("K,N,masked", [(K, N, m) for (K, N) in sorted(set(STACK["shapes"])) for m in (True, False)])
def test_llama7b_stack_layers_sampled(K, N, masked):
    """A masked block's layer (rank 64) and an unmasked one (plain W4), both
    per-output-channel symmetric, at the mixed step's prefill and decode sizes."""
    r = STACK["r"] if masked else 0
    L, OL = _layer(N, K, r, K, True, seed=3 * N + K + r)
    _check(L, OL, STACK["prefill_M"][0], K, N, "prefill", 96, 11, STACK["outlier_frac"])
    _check(L, OL, STACK["decode_M"][0], K, N, "decode", 128, 12, STACK["outlier_frac"])


@pytest.mark.parametrize("K,N", P7["shapes"])
def test_llama7b_prefill_largest_chunk_sampled(K, N):
    """M = 8192, the prefill workload's largest chunk."""
    M = max(P7["prefill_M"])
    L, OL = _layer(N, K, P7["r"], P7["G"], P7["sym"], seed=5 * N + K)
    _check(L, OL, M, K, N, "prefill", 48, 8192 + K, P7["outlier_frac"])
