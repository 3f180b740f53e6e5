"""The Python binding's own argument checks, on CPU: the shapes and dtypes of
x and y that the C ABI (plain pointers) cannot see are refused before any
pointer reaches the library."""
import pytest
import torch

from quantized_gemm_error_gb300 import spear


def _layer(N=128, K=256):
    return spear.W4Layer(N, K, 128, True, torch.zeros(N, K // 2, dtype=torch.uint8),
                         torch.zeros(N, K // 128, dtype=torch.float16))


@pytest.mark.parametrize("call", [spear.spear_linear_decode, spear.spear_linear_prefill])
def test_tokens_must_be_bf16_rows_of_width_k(call):
    L = _layer()
    with pytest.raises(ValueError, match="bfloat16"):
        call(L, torch.zeros(4, 256, dtype=torch.float16))
    with pytest.raises(ValueError, match="256"):
        call(L, torch.zeros(4, 128, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        call(L, torch.zeros(256, dtype=torch.bfloat16))


@pytest.mark.parametrize("call", [spear.spear_linear_decode, spear.spear_linear_prefill])
def test_output_must_match_the_requested_type_and_shape(call):
    L = _layer()
    x = torch.zeros(4, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="float32"):
        call(L, x, y=torch.zeros(4, 128, dtype=torch.bfloat16), out_dtype=spear.OUT_F32)
    with pytest.raises(ValueError, match="128"):
        call(L, x, y=torch.zeros(4, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="out_dtype"):
        call(L, x, out_dtype=7)


def test_noalloc_decode_checks_its_output_too():
    L = _layer()
    x = torch.zeros(2, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="bfloat16"):
        spear.spear_linear_decode_noalloc(L, x, y=torch.zeros(2, 128, dtype=torch.float32))


def test_layer_tensors_are_checked():
    import dataclasses
    L = _layer()
    L.check()
    bad = [dict(qweight=torch.zeros(128, 64, dtype=torch.uint8)),           # [N][K/2] is [128][128]
           dict(scales=torch.zeros(128, 2, dtype=torch.float32)),
           dict(symmetric=False),                                          # zero points missing
           dict(group_size=96)]
    for kw in bad:
        with pytest.raises(ValueError):
            dataclasses.replace(L, **kw).check()
    bf = lambda *s: torch.zeros(*s, dtype=torch.bfloat16)
    C = dataclasses.replace(L, rank=16, A=bf(16, 256), B=bf(128, 16), w_g=bf(256))
    C.check()
    with pytest.raises(ValueError, match="B"):
        dataclasses.replace(C, B=bf(16, 128)).check()                      # transposed
    with pytest.raises(ValueError, match="w_g"):
        dataclasses.replace(C, w_g=None).check()
    f32 = lambda *s: torch.zeros(*s, dtype=torch.float32)
    V = dataclasses.replace(C, w_g=None, gate_w1=f32(8, 16), gate_c1=f32(8), gate_w2=f32(16, 8), gate_c2=f32(16))
    V.check()
    with pytest.raises(ValueError, match="gate_w2"):
        dataclasses.replace(V, gate_w2=f32(8, 16)).check()
    dataclasses.replace(C, comp_enabled=False, A=None, B=None, w_g=None).check()   # plain layer: no factors
