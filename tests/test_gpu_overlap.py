"""Overlapped decode launches (spear_set_launch_overlap): a chain of decode
calls in which every call reads the previous call's output must give the same
bits with and without overlap, eagerly and inside a captured CUDA graph, on
both decode kernels (M <= 16 and M >= 17)."""
import pytest
import torch

from spear_testutil import gpu_layer, make_layer, make_tokens, to_dev_u16

pytestmark = pytest.mark.gpu


def _spear():
    from quantized_gemm_error_gb300 import spear
    return spear


def _chain(sp, layers, x0, ws, stream, graph=False):
    """y_i = layer_i(y_{i-1}) on one stream; returns every output."""
    outs = [torch.empty(x0.shape[0], L.N, dtype=torch.bfloat16, device="cuda") for L in layers]

    def run():
        x = x0
        for L, y in zip(layers, outs):
            sp.spear_linear_decode(L, x, y=y, workspace=ws, stream=stream)
            x = y
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run()
        g.replay()
    else:
        with torch.cuda.stream(stream):
            run()
    torch.cuda.synchronize()
    assert sp.spear_get_device_status() == 0
    return [o.clone() for o in outs]


@pytest.mark.parametrize("M", [3, 48])
def test_overlapped_chain_is_bit_identical(M):
    sp = _spear()
    K = 1024
    layers = []
    for i in range(5):
        lay, rng = make_layer(K, K, 32, seed=300 + i)
        layers.append(gpu_layer(lay, 128, False))
    x0 = to_dev_u16(make_tokens(rng, M, K), torch.bfloat16)
    ws = sp.new_workspace(max(sp.spear_decode_workspace_bytes(L, M) for L in layers), "cuda")
    stream = torch.cuda.Stream()
    sp.spear_set_launch_overlap(False)
    ref = _chain(sp, layers, x0, ws, stream)
    try:
        sp.spear_set_launch_overlap(True)
        eager = _chain(sp, layers, x0, ws, stream)
        graphed = _chain(sp, layers, x0, ws, stream, graph=True)
    finally:
        sp.spear_set_launch_overlap(False)
    for a, b, c in zip(ref, eager, graphed):
        assert torch.equal(a, b)
        assert torch.equal(a, c)
    assert not ws[:16].any(), "workspace sync words not left zeroed"
