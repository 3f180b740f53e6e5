"""The bounds-checked build (-DSPEAR_DEBUG_CHECKS, lib/libspear_debug.so):
every kernel checks the indices it forms -- tile and K-slice ranges, ring
slots, global addresses of the weight stream, shared-memory extents,
workspace and output indices -- and a failed check records SPEAR_ERR_BOUNDS
in its status word (no trap).  The small parity cases run through that build
in a child process (a process loads one build of the library): every call
must leave the status at 0 and still match the oracle.

Source: SPEAR explainer, Technical Summary 2.1 A and 2.2 A (the layer and its
decode / prefill kernels); the checks are this library's."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CHILD = r"""
import sys
sys.path[:0] = [ROOT, HERE]
import numpy as np
import torch
import oracle
from quantized_gemm_error_gb300 import build, spear
spear.load(build.DEBUG_LIB_PATH)
from spear_testutil import check_close, gpu_layer, make_layer, make_tokens, oracle_layer, to_dev_u16

def status_ok(what):
    s = spear.spear_get_device_status()
    assert s == 0, f"{what}: device status {spear.STATUS_NAMES.get(s, s)}"

# packing: compared bit for bit with the oracle
for (N, K, G, sym) in [(64, 256, 128, True), (192, 384, 128, False), (128, 1024, 1024, False)]:
    lay, _ = make_layer(N, K, 0, seed=N + K)
    q, s, z = spear.spear_pack_w4(torch.from_numpy(lay.W).cuda(), G, sym)
    torch.cuda.synchronize()
    status_ok(f"pack {N}x{K}")
    qo, so, zo = oracle.quantize_pack(lay.W, G, sym)
    assert (q.cpu().numpy() == qo).all()

# decode: both warp-level token tiles, staged and L1 tokens, the tensor-core kernel
for (N, K, G, sym, r, M) in [(64, 128, 128, True, 16, 1), (192, 384, 128, False, 16, 3),
                             (1024, 1024, 1024, True, 16, 16), (512, 2048, 128, False, 32, 9),
                             (512, 1024, 128, False, 32, 24), (256, 2048, 2048, True, 64, 32),
                             (320, 1152, 128, False, 64, 33), (256, 1024, 1024, False, 32, 64),
                             (1024, 1024, 128, True, 0, 5)]:
    lay, rng = make_layer(N, K, r, seed=100 + N + M)
    x = make_tokens(rng, M, K, outlier_frac=0.01)
    L = gpu_layer(lay, G, sym)
    ref = oracle.linear(oracle_layer(lay, G, sym), x, nthreads=8)
    y = spear.spear_linear_decode(L, to_dev_u16(x, torch.bfloat16), out_dtype=spear.OUT_F32)
    torch.cuda.synchronize()
    status_ok(f"decode {N}x{K} M={M}")
    check_close(y, ref)

# prefill: 128- and 256-token tiles, ragged M and N, K split, both compensator modes
for (N, K, G, sym, r, M) in [(256, 256, 128, False, 0, 200), (320, 2048, 128, False, 64, 257),
                             (1024, 1024, 1024, True, 32, 512), (2560, 512, 128, False, 32, 2000)]:
    lay, rng = make_layer(N, K, r, seed=41 + N + M + r)
    x = make_tokens(rng, M, K, outlier_frac=0.01)
    L = gpu_layer(lay, G, sym)
    ref = oracle.linear(oracle_layer(lay, G, sym), x, nthreads=8)
    for mode in (spear.PREFILL_FUSED, spear.PREFILL_STREAM):
        y = spear.spear_linear_prefill(L, to_dev_u16(x, torch.bfloat16), out_dtype=spear.OUT_F32, mode=mode,
                                       stream_aux=torch.cuda.Stream())
        torch.cuda.synchronize()
        status_ok(f"prefill {N}x{K} M={M} mode={mode}")
        check_close(y, ref)
print("debug-checks: all cases clean")
"""


def test_small_parity_cases_pass_the_index_checks():
    from quantized_gemm_error_gb300 import build
    build.build_library(debug=True)
    code = CHILD.replace("ROOT", repr(ROOT)).replace("HERE", repr(HERE))
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    assert "all cases clean" in res.stdout
