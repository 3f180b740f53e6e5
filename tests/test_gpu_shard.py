"""GPU parity for the column-parallel split (quantized_gemm_error_gb300/shard.py):
each rank's shard, run through the library's decode and prefill calls on one
GPU in turn, gives its slice of y within the layer's tolerance of the oracle,
and the slices together cover every output.  (Deployed, each shard runs on
a GPU of its own; the test runs them one after another on one GPU.)"""
import pytest
import torch

import oracle
from spear_testutil import check_close, gpu_layer, make_layer, make_tokens, oracle_layer, to_dev_u16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K,G,sym,r,world,M,path", [
    (1024, 1024, 128, False, 32, 2, 4, "decode"),      # warp-level decode
    (1024, 1024, 128, False, 32, 3, 40, "decode"),     # tensor-core decode, uneven ranges
    (1024, 1024, 1024, True, 16, 2, 300, "prefill"),   # per-channel scales
    (1536, 2048, 128, False, 64, 4, 512, "prefill"),   # group scales, rank 64
])
def test_shards_give_their_slice_of_y(N, K, G, sym, r, world, M, path):
    from quantized_gemm_error_gb300 import spear
    from quantized_gemm_error_gb300.shard import column_ranges, column_shard
    lay, rng = make_layer(N, K, r, seed=90 + N + M)
    x_bits = make_tokens(rng, M, K, outlier_frac=0.01)
    ref = oracle.linear(oracle_layer(lay, G, sym), x_bits, nthreads=8)
    L = gpu_layer(lay, G, sym)
    x = to_dev_u16(x_bits, torch.bfloat16)
    ys = []
    for k in range(world):
        S = column_shard(L, k, world)
        n0, n1 = column_ranges(N, world)[k]
        if path == "decode":
            y = spear.spear_linear_decode(S, x, out_dtype=1)
        else:
            y = spear.spear_linear_prefill(S, x, out_dtype=1)
        torch.cuda.synchronize()
        assert spear.spear_get_device_status() == 0
        assert tuple(y.shape) == (M, n1 - n0)
        check_close(y, ref[:, n0:n1], f"rank {k} of {world}")
        ys.append(y)
    assert sum(y.shape[1] for y in ys) == N
