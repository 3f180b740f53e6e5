"""The decode entry point for callers that cannot allocate device memory.

Plugins hosted by a framework that owns the device allocator, runtimes that
plan every buffer before serving and forbid allocation afterwards, and code on
latency-critical paths where an allocation could synchronise the device all
need a decode call that takes only inputs and outputs.  spear_linear_decode_noalloc
keeps its scratch in a fixed array inside the library instead of a caller
workspace.  Its output must match spear_linear_decode's within the parity
tolerance, on two calls in a row (the second reuses what the first left in the
shared scratch), and the largest workload shape must fit that scratch.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes when run alone.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from spear_testutil import check_close, gpu_layer, make_layer, make_tokens, to_dev_u16

pytestmark = pytest.mark.gpu


def _spear():
    from quantized_gemm_error_gb300 import spear
    return spear


@pytest.mark.parametrize("N,K,G,sym,r,M", [
    (1024, 2048, 128, False, 32, 4),        # group-128 asymmetric, rank 32
    (1024, 1024, 1024, True, 16, 1),        # per-channel symmetric, rank 16
    (4096, 4096, 128, False, 32, 16),       # Llama-7B square linear
])
def test_noalloc_decode_matches_workspace_decode(N, K, G, sym, r, M):
    sp = _spear()
    lay, rng = make_layer(N, K, r, seed=90 + N + M)
    L = gpu_layer(lay, G, sym)
    for out_dtype, dt in ((sp.OUT_BF16, torch.bfloat16), (sp.OUT_F32, torch.float32)):
        x = to_dev_u16(make_tokens(rng, M, K, outlier_frac=0.01), torch.bfloat16)
        ref = sp.spear_linear_decode(L, x, out_dtype=out_dtype)
        torch.cuda.synchronize()
        ref64 = ref.float().cpu().numpy().astype(np.float64)
        for call in range(2):                    # two calls in a row on the shared scratch
            y = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
            sp.spear_linear_decode_noalloc(L, x, y=y, out_dtype=out_dtype)
            torch.cuda.synchronize()
            assert sp.spear_get_device_status() == 0
            check_close(y, ref64, f"noalloc call {call + 1}")


def test_noalloc_decode_alternating_shapes():
    """Calls with different layers and token counts back to back share the one scratch."""
    sp = _spear()
    cases = []
    for i, (N, K, M) in enumerate([(1024, 1024, 3), (512, 2048, 64), (1024, 1024, 1)]):
        lay, rng = make_layer(N, K, 32, seed=95 + i)
        L = gpu_layer(lay, 128, False)
        x = to_dev_u16(make_tokens(rng, M, K), torch.bfloat16)
        cases.append((L, x, sp.spear_linear_decode(L, x, out_dtype=sp.OUT_F32)))
    torch.cuda.synchronize()
    for L, x, ref in cases + cases:
        y = torch.empty(ref.shape, dtype=torch.float32, device="cuda")
        sp.spear_linear_decode_noalloc(L, x, y=y, out_dtype=sp.OUT_F32)
        torch.cuda.synchronize()
        check_close(y, ref.cpu().numpy().astype(np.float64), "noalloc")
    assert sp.spear_get_device_status() == 0


def test_noalloc_serves_the_largest_workload_shape():
    """28672 x 8192 (70B down-projection shape) at M = 64 fits the built-in
    scratch and matches the workspace path bit for bit (same kernel, same split)."""
    sp = _spear()
    N, K, r, M = 8192, 28672, 64, 64
    lay, rng = make_layer(N, K, r, seed=97)
    L = gpu_layer(lay, 128, False)
    assert sp.spear_decode_workspace_bytes(L, M) <= 8 << 20
    x = to_dev_u16(make_tokens(rng, M, K, outlier_frac=0.01), torch.bfloat16)
    ref = sp.spear_linear_decode(L, x)
    y = torch.empty_like(ref)
    sp.spear_linear_decode_noalloc(L, x, y=y)
    torch.cuda.synchronize()
    assert sp.spear_get_device_status() == 0
    assert torch.equal(y, ref)


_FIRST_CALL_ON_SIDE_STREAM = r"""
import sys
sys.path[:0] = [ROOT, os.path.join(ROOT, "tests")]
import numpy as np, torch
from spear_testutil import check_close, gpu_layer, make_layer, make_tokens, to_dev_u16
from quantized_gemm_error_gb300 import spear as sp
torch.cuda.set_device(0)
lay, rng = make_layer(2048, 4096, 32, seed=99)
L = gpu_layer(lay, 128, False)
x = to_dev_u16(make_tokens(rng, 12, 4096, outlier_frac=0.01), torch.bfloat16)
torch.cuda.synchronize()
side = torch.cuda.Stream()                       # a non-blocking stream
y = torch.full((12, 2048), float("nan"), dtype=torch.float32, device="cuda")
with torch.cuda.stream(side):
    sp.spear_linear_decode_noalloc(L, x, y=y, out_dtype=sp.OUT_F32, stream=side)   # first call of the process
    ref = sp.spear_linear_decode(L, x, out_dtype=sp.OUT_F32, stream=side)
side.synchronize()
assert sp.spear_get_device_status() == 0
check_close(y, ref.cpu().numpy().astype(np.float64), "first noalloc call on a side stream")
print("ok")
"""


def test_noalloc_first_call_of_a_process_on_a_side_stream():
    """The first no-alloc call of a fresh process, issued on a non-blocking
    stream, gives the workspace path's output: its one-time set-up is ordered
    before the kernel whatever stream the caller uses."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = f"import os\nROOT = {root!r}\n" + _FIRST_CALL_ON_SIDE_STREAM
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert res.returncode == 0 and "ok" in res.stdout, res.stdout[-2000:] + res.stderr[-4000:]
