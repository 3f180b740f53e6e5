"""The decoder-block stack helper on the GPU: a two-block stack (one plain W4
block, one with rank-64 compensators), per-output-channel symmetric int4 at
the Llama-7B shapes.  Graph replay reproduces the eager calls bit for bit,
and sampled outputs of a plain and a compensated layer match the oracle on
both paths (prefill M = 1056, decode M = 32).

Source: SPEAR explainer, Technical Summary 2.1 A/B and 2.2 A."""
import pytest
import torch

import oracle
from quantized_gemm_error_gb300.inputs import make_layer
from spear_testutil import check_close, oracle_layer, sample_columns

pytestmark = pytest.mark.gpu


def test_two_block_stack_graph_matches_eager_and_oracle():
    from quantized_gemm_error_gb300 import spear
    from quantized_gemm_error_gb300.stack import StackStep, build_stack
    dev = torch.device("cuda", 0)
    ranks = [0, 64]
    layers = build_stack(ranks, dev, seed=5, recipe="numpy")
    step = StackStep(layers, 1056, 32, dev, seed=6)
    step.capture()
    torch.cuda.synchronize()
    eager_p = [y.clone() for y in step.yp]
    eager_d = [y.clone() for y in step.yd]
    for y in step.yp + step.yd:
        y.zero_()
    step.replay("prefill")
    step.replay("decode")
    torch.cuda.synchronize()
    assert spear.spear_get_device_status() == 0
    for a, b in zip(eager_p + eager_d, step.yp + step.yd):
        assert torch.equal(a, b)
    # oracle on sampled rows: block 0 "gate" (plain) and block 1 "down" (compensated)
    for idx in (4, 7 + 6):
        sl = layers[idx]
        lay, _ = make_layer(sl.N, sl.K, ranks[sl.block], seed=5 + 1000 * sl.block + idx % 7)
        OL = oracle_layer(lay, sl.K, True)
        cols = sample_columns(sl.N, 64, seed=idx)
        ci = torch.from_numpy(cols).cuda()
        ref_p = oracle.linear(OL, step.xp_bits[sl.K], n_idx=cols, nthreads=8)
        ref_d = oracle.linear(OL, step.xd_bits[sl.K], n_idx=cols, nthreads=8)
        check_close(step.yp[idx][:, ci], ref_p, f"{sl.name}{sl.block} prefill")
        check_close(step.yd[idx][:, ci], ref_d, f"{sl.name}{sl.block} decode")
