"""CPU-only checks of the C ABI: the library loads, exports every symbol that
include/spear.h declares, and its host-only logic (argument checks, packed
sizes, module selection) behaves as specified.  No compute call touches a GPU.
"""
import ctypes
import json
import os
import re

import numpy as np
import pytest

import oracle
from quantized_gemm_error_gb300 import build, spear

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = json.load(open(os.path.join(ROOT, "tests", "golden", "worked_examples.json")))


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return spear.load()


def declared_symbols():
    hdr = open(os.path.join(ROOT, "include", "spear.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return sorted(set(re.findall(r"\b(spear_[a-z0-9_]+)\s*\(", hdr)))


def test_exports_every_declared_symbol(lib):
    decl = declared_symbols()
    assert decl, "no declarations found"
    assert sorted(spear.EXPORTS) == decl
    for name in decl:
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert lib.spear_status_string(0) == b"SPEAR_OK"
    assert lib.spear_status_string(5) == b"SPEAR_ERR_TIMEOUT"
    assert spear.version().count(".") == 2


def test_pack_sizes(lib):
    assert spear.spear_pack_w4_sizes(4096, 11008, 128, False) == (4096 * 11008 // 2, 4096 * 86 * 2, 4096 * 43)
    assert spear.spear_pack_w4_sizes(1024, 1024, 1024, True) == (1024 * 512, 1024 * 2, 0)
    for args in [(4096, 4000, 128, True), (100, 4096, 128, True), (4096, 4096, 64, True), (0, 128, 128, True)]:
        with pytest.raises(spear.SpearError) as e:
            spear.spear_pack_w4_sizes(*args)
        assert e.value.status == 1
    # sizes agree with the oracle's packed format
    assert spear.spear_pack_w4_sizes(64, 1024, 128, False) == oracle.packed_sizes(64, 1024, 128, False)


def test_invalid_layer_rejected_before_any_device_work(lib):
    L = spear._Layer(N=64, K=128, group_size=128, symmetric=1, qweight=None, scales=None, zeros=None, rank=16,
                     A=None, B=None, w_g=None, b_g=0.0, alpha=1.0, comp_enabled=1)
    n = ctypes.c_size_t()
    assert lib.spear_decode_workspace_bytes(ctypes.byref(L), 1, ctypes.byref(n)) == 1
    assert b"NULL" in lib.spear_last_error()
    L.qweight, L.scales = 16, 32
    L.rank = 24
    assert lib.spear_decode_workspace_bytes(ctypes.byref(L), 1, ctypes.byref(n)) == 1
    assert b"rank" in lib.spear_last_error()
    L.rank, L.qweight = 16, 17                                # misaligned
    assert lib.spear_decode_workspace_bytes(ctypes.byref(L), 1, ctypes.byref(n)) == 1
    L.qweight, L.A, L.B, L.w_g = 16, 48, 64, 80
    assert lib.spear_decode_workspace_bytes(ctypes.byref(L), 65, ctypes.byref(n)) == 1   # M > 64
    assert lib.spear_linear_prefill(ctypes.byref(L), None, 8, None, 0, 0, None, 0, None, None) == 1
    assert lib.spear_linear_decode(ctypes.byref(L), 16, 1, 32, 7, None, 0, None) == 1      # out_dtype
    # the vector gate: hidden width in [1, 32], its four buffers present and aligned
    L.gate_hidden = 33
    assert lib.spear_decode_workspace_bytes(ctypes.byref(L), 1, ctypes.byref(n)) == 1
    assert b"gate_hidden" in lib.spear_last_error()
    L.gate_hidden = 8
    assert lib.spear_decode_workspace_bytes(ctypes.byref(L), 1, ctypes.byref(n)) == 1
    assert b"vector-gate buffers are NULL" in lib.spear_last_error()
    L.gate_w1, L.gate_c1, L.gate_w2, L.gate_c2 = 96, 112, 128, 148           # gate_c2 misaligned
    assert lib.spear_decode_workspace_bytes(ctypes.byref(L), 1, ctypes.byref(n)) == 1
    assert b"aligned" in lib.spear_last_error()


def test_layer_select_matches_worked_example_and_oracle(lib):
    ex = GOLDEN["layer_select"]
    for case in ex["cases"]:
        m, r = spear.spear_layer_select_mask(ex["damage"], ex["cost"], case["budget"], case["rank_min"],
                                             case["rank_max"])
        assert m.tolist() == case["mask"] and r.tolist() == case["rank"]
    rng = np.random.default_rng(11)
    for trial in range(200):
        L = int(rng.integers(1, 40))
        d = (rng.random(L) ** rng.uniform(0.5, 6)).astype(np.float32)
        if trial % 7 == 0:
            d[rng.random(L) < 0.5] = 0
        c = rng.uniform(100, 5000, L).astype(np.float32)
        budget = float(rng.uniform(1e3, 2e6))
        rmin, rmax = int(rng.choice([1, 16, 17])), int(rng.choice([16, 64, 128, 130]))
        if rmax < rmin:
            rmin, rmax = rmax, rmin
        try:
            mo, ro = oracle.layer_select_mask(d, c, budget, rmin, rmax)
        except ValueError:
            with pytest.raises(spear.SpearError):
                spear.spear_layer_select_mask(d, c, budget, rmin, rmax)
            continue
        mg, rg = spear.spear_layer_select_mask(d, c, budget, rmin, rmax)
        assert (mo == mg).all() and (ro == rg).all()


def test_layer_select_rejects_bad_input(lib):
    with pytest.raises(spear.SpearError):
        spear.spear_layer_select_mask([1.0, -1.0], [1.0, 1.0], 100.0, 16, 64)
    with pytest.raises(spear.SpearError):
        spear.spear_layer_select_mask([1.0, 1.0], [1.0, 0.0], 100.0, 16, 64)
    with pytest.raises(spear.SpearError):
        spear.spear_layer_select_mask([1.0], [1.0], 100.0, 17, 31)     # no multiple of 16 in range
