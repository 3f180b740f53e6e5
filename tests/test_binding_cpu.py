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
