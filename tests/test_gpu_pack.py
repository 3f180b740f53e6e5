"""GPU parity for spear_pack_w4: packed codes, fp16 scales and uint4 zero
points must equal the oracle's bytes exactly (RTN int4, SPEAR explainer,
Technical Summary 3.1)."""
import numpy as np
import pytest
import torch

import oracle
from quantized_gemm_error_gb300.inputs import make_layer

pytestmark = pytest.mark.gpu


def _pack_both(W, G, sym):
    from quantized_gemm_error_gb300 import spear
    q, s, z = spear.spear_pack_w4(torch.from_numpy(W).cuda(), G, sym)
    torch.cuda.synchronize()
    assert spear.spear_get_device_status() == 0
    qo, so, zo = oracle.quantize_pack(W, G, sym)
    return (q.cpu().numpy(), s.cpu().view(torch.int16).numpy().view(np.uint16),
            None if z is None else z.cpu().numpy()), (qo, so, zo)


@pytest.mark.parametrize("N,K,G,sym", [
    (64, 128, 128, True), (64, 128, 128, False),          # one tile, one group
    (1024, 1024, 1024, True),                             # per-channel, 1024^2
    (192, 11008, 128, False),                             # 86 groups: odd number of zero pairs
    (256, 4096, 4096, False),                             # per-channel asymmetric
    (128, 28672, 128, True),
])
def test_pack_bit_exact(N, K, G, sym):
    lay, _ = make_layer(N, K, 0, seed=N + K)
    W = lay.W
    W[3, :] = 0.0                                         # all-zero row
    W[5, :G] *= 1000.0                                    # one wide group
    W[7, 1] = 2.0 ** -30                                  # tiny values -> fp16 subnormal scale
    W[9, ::2] = -W[9, 1::2]
    (q, s, z), (qo, so, zo) = _pack_both(W, G, sym)
    assert (q == qo).all()
    assert (s == so).all()
    if not sym:
        assert (z == zo).all()


def test_pack_exact_grid_and_ties():
    """Values exactly halfway between grid points exercise round-half-to-even."""
    rng = np.random.default_rng(12)
    N, K, G = 64, 256, 128
    s = np.float32(0.125)
    q = rng.integers(-7, 8, size=(N, K)).astype(np.float32)
    q[:, ::G] = 7
    W = (q * s).astype(np.float32)
    W[:, 5::9] += s / 2                                   # exact ties
    (qg, sg, _), (qo, so, _) = _pack_both(W, G, True)
    assert (qg == qo).all() and (sg == so).all()


def test_pack_reports_non_finite():
    from quantized_gemm_error_gb300 import spear
    W = torch.zeros(64, 128, device="cuda")
    W[10, 3] = float("inf")
    spear.spear_pack_w4(W, 128, True)
    assert spear.spear_get_device_status() == 1
    assert spear.spear_get_device_status() == 0           # read clears it
