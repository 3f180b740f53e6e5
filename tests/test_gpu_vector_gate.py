"""GPU parity of the pages' vector gate (Technical Summary 2.1 A: effective
weight W + alpha B diag(gamma(A x)) A, gamma a bottleneck MLP; read as
gamma(t) = sigmoid(W2 relu(W1 t + c1) + c2)) against the oracle's
linear_vector_gate: decode on the warp-level kernel (1, 5, 12 tokens) and the
tensor-core kernel (20-64 tokens, ranks 16, 32 and 64), prefill on 128- and 256-token tiles in
both modes; no w_g is given."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from spear_testutil import check_close, gpu_layer, make_layer, make_tokens, oracle_layer, to_dev_u16

pytestmark = pytest.mark.gpu


def _gate(rng, r, h):
    W1 = (rng.standard_normal((h, r)) * (3.0 / np.sqrt(r))).astype(np.float32)
    c1 = (rng.standard_normal(h) * 0.1).astype(np.float32)
    W2 = (rng.standard_normal((r, h)) * (1.0 / np.sqrt(h))).astype(np.float32)
    c2 = rng.standard_normal(r).astype(np.float32)
    return W1, c1, W2, c2


def _layers(N, K, G, sym, r, h, seed):
    lay, rng = make_layer(N, K, r, seed=seed)
    W1, c1, W2, c2 = _gate(np.random.default_rng(seed + 1), r, h)
    L = gpu_layer(lay, G, sym)
    dev = lambda a: torch.from_numpy(a).cuda()
    L = dataclasses.replace(L, w_g=None, gate_w1=dev(W1), gate_c1=dev(c1), gate_w2=dev(W2), gate_c2=dev(c2))
    return L, oracle_layer(lay, G, sym), (W1, c1, W2, c2), rng


@pytest.mark.parametrize("N,K,G,sym,r,h,M", [
    (512, 1024, 128, False, 32, 8, 1),
    (512, 1024, 128, False, 32, 8, 5),       # tokens staged in shared memory
    (256, 2048, 128, False, 16, 4, 12),      # two token tiles
    (320, 1152, 128, False, 64, 16, 24),     # tensor-core kernel, 32 token rows
    (256, 1024, 1024, True, 32, 32, 64),     # tensor-core kernel, per-channel scales
    # tensor-core kernel: the gate's lanes per token and pieces per lane for
    # each rank, hidden widths that are not multiples of 8
    (512, 1024, 128, False, 16, 5, 40),      # 2 lanes per token, 2 pieces each
    (384, 2048, 128, False, 64, 9, 64),      # 8 pieces per lane, two hidden chunks
    (256, 1024, 128, False, 16, 3, 20),      # 4 lanes per token, 1 piece each
    (320, 1536, 128, True, 32, 12, 33),      # 2 lanes per token, 4 pieces each
])
def test_decode_vector_gate_matches_oracle(N, K, G, sym, r, h, M):
    from quantized_gemm_error_gb300 import spear
    L, OL, g, rng = _layers(N, K, G, sym, r, h, seed=200 + N + M)
    x = make_tokens(rng, M, K, outlier_frac=0.01)
    ref, gam = oracle.linear_vector_gate(OL, x, *g, nthreads=8)
    assert 0.02 < gam.mean() < 0.98 and gam.std() > 0.05           # the gate really varies
    y = spear.spear_linear_decode(L, to_dev_u16(x, torch.bfloat16), out_dtype=1)
    torch.cuda.synchronize()
    assert spear.spear_get_device_status() == 0
    check_close(y, ref)


@pytest.mark.parametrize("N,K,G,sym,r,h,M", [
    (512, 1024, 128, False, 32, 8, 300),     # 128-token tiles
    (2560, 512, 128, False, 32, 8, 2000),    # 256-token tiles: the correction joins the main accumulators
    (512, 1024, 1024, True, 64, 16, 200),    # per-channel scales
])
@pytest.mark.parametrize("mode", [1, 2])
def test_prefill_vector_gate_matches_oracle(N, K, G, sym, r, h, M, mode):
    from quantized_gemm_error_gb300 import spear
    L, OL, g, rng = _layers(N, K, G, sym, r, h, seed=300 + N + M)
    x = make_tokens(rng, M, K, outlier_frac=0.01)
    ref, _ = oracle.linear_vector_gate(OL, x, *g, nthreads=8)
    y = spear.spear_linear_prefill(L, to_dev_u16(x, torch.bfloat16), out_dtype=1, mode=mode,
                                   stream_aux=torch.cuda.Stream())
    torch.cuda.synchronize()
    assert spear.spear_get_device_status() == 0
    check_close(y, ref)


def test_vector_gate_hidden_width_is_checked():
    from quantized_gemm_error_gb300 import spear
    L, _, g, rng = _layers(256, 512, 128, False, 16, 4, seed=7)
    h = 33                                                   # one past the library's limit
    big = dict(gate_w1=torch.zeros(h, 16, device="cuda"), gate_c1=torch.zeros(h, device="cuda"),
               gate_w2=torch.zeros(16, h, device="cuda"), gate_c2=torch.zeros(16, device="cuda"))
    with pytest.raises(spear.SpearError):
        spear.spear_linear_decode(dataclasses.replace(L, **big), to_dev_u16(make_tokens(rng, 1, 512),
                                                                              torch.bfloat16))


@pytest.mark.parametrize("M,path", [(5, "decode"), (40, "decode"), (300, "prefill")])
def test_vector_gate_activations_of_any_magnitude(M, path):
    """Tokens up to ~1e6 (beyond fp16) with the vector gate: the gate's
    down-projection runs on the bf16 tokens, the main term through the fp16
    launches' scaling (staged tokens, the tensor-core kernel's fp32 path for
    overflowed tokens, prefill's power-of-two token scaling)."""
    from quantized_gemm_error_gb300 import spear
    from quantized_gemm_error_gb300.inputs import f32_to_bf16_bits
    from spear_testutil import bf16_bits_to_f32
    N, K = 512, 1024
    L, OL, g, rng = _layers(N, K, 128, False, 32, 8, seed=500 + M)
    x = bf16_bits_to_f32(make_tokens(rng, M, K, outlier_frac=0.01)).reshape(M, K)
    row_scale = np.ones(M, np.float32)
    row_scale[0::3] = 3.0e4
    x = f32_to_bf16_bits(x * row_scale[:, None])
    ref, _ = oracle.linear_vector_gate(OL, x, *g, nthreads=8)
    xd = to_dev_u16(x, torch.bfloat16)
    if path == "decode":
        y = spear.spear_linear_decode(L, xd, out_dtype=1)
    else:
        y = spear.spear_linear_prefill(L, xd, out_dtype=1, mode=spear.PREFILL_FUSED)
    torch.cuda.synchronize()
    assert spear.spear_get_device_status() == 0
    check_close(y, ref)
