"""SLO-constrained chunk selection (Technical Summary 2.2 C) on the host:
spear_chunk_select against closed forms and the oracle's plain restatement."""
import numpy as np
import pytest

import oracle


def _spear():
    from quantized_gemm_error_gb300 import spear
    spear.load()
    return spear


def test_linear_curves_closed_form():
    # every layer: prefill us = 50 + 0.4 M, decode us = 8 + 0.1 M; 10 layers, D = 32
    pre = [([256, 4096], [50 + 0.4 * 256, 50 + 0.4 * 4096])] * 10
    dec = [([1, 64], [8.1, 14.4])] * 10
    C, step = _spear().spear_chunk_select(pre, dec, 32, [0, 256, 512, 1024, 2048], 3000.0)
    # 10 (50 + 0.4 (C + 32)) <= 3000  ->  C <= 668: the largest listed is 512
    assert C == 512 and step == pytest.approx(10 * (50 + 0.4 * 544), rel=1e-6)
    C0, s0 = _spear().spear_chunk_select(pre, dec, 32, [0, 256], 50.0)
    assert C0 == 0 and s0 == pytest.approx(10 * (8 + 0.1 * 32), rel=1e-6)   # decode-only step


def test_interpolation_and_extrapolation():
    pre = [([256, 1024, 4096], [100.0, 300.0, 1500.0])]
    dec = [([16], [20.0])]
    sp = _spear()
    for D, C, want in [(0, 640, 200.0), (0, 128, 66.6667), (0, 8192, 3100.0), (16, 0, 20.0)]:
        got = sp.spear_chunk_select(pre, dec, D, [C], 1e9)
        assert got[0] == C and got[1] == pytest.approx(want, rel=1e-4)


def test_no_choice_fits_returns_the_smallest():
    pre = [([256, 512], [1000.0, 2000.0])]
    dec = [([1, 8], [500.0, 600.0])]
    C, step = _spear().spear_chunk_select(pre, dec, 4, [256, 1024, 0], 100.0)
    assert C == 0 and step == pytest.approx(500.0 + 100.0 * 3 / 7, rel=1e-6)


def test_monotone_in_target_and_in_compensator_density():
    rng = np.random.default_rng(0)
    Ms = [256, 512, 1024, 2048, 4096]
    plain = [(Ms, list(np.cumsum(rng.uniform(20, 60, 5))))] * 7
    comp = [(Ms, [u * 1.2 for u in plain[0][1]])] * 7
    dec = [([1, 32, 64], [5.0, 8.0, 12.0])] * 7
    choices = [0, 128, 256, 512, 1024, 2048, 4096]
    sp = _spear()
    last = -1
    for target in np.linspace(10, 3000, 25):
        C, _ = sp.spear_chunk_select(plain, dec, 32, choices, target)
        assert C >= last
        last = C
    for target in (400.0, 900.0, 1800.0):
        lo, _ = sp.spear_chunk_select(comp, dec, 32, choices, target)
        hi, _ = sp.spear_chunk_select(plain, dec, 32, choices, target)
        assert lo <= hi                                   # more compensators, never a larger chunk


def test_matches_the_oracle_on_random_curves():
    rng = np.random.default_rng(1)
    sp = _spear()
    for trial in range(200):
        L = int(rng.integers(1, 12))
        pre, dec = [], []
        for _ in range(L):
            n = int(rng.integers(1, 6))
            Ms = np.sort(rng.choice(np.arange(16, 8192), size=n, replace=False)).tolist()
            pre.append((Ms, rng.uniform(0, 500, n).astype(np.float32).tolist()))
            n2 = int(rng.integers(1, 5))
            Md = np.sort(rng.choice(np.arange(1, 128), size=n2, replace=False)).tolist()
            dec.append((Md, rng.uniform(0, 50, n2).astype(np.float32).tolist()))
        D = int(rng.integers(0, 65))
        choices = sorted(set(rng.choice([0, 64, 128, 256, 512, 1024, 2048, 4096], size=4).tolist()))
        target = float(rng.uniform(0, 5000))
        got = sp.spear_chunk_select(pre, dec, D, choices, target)
        ref = oracle.chunk_select(pre, dec, D, choices, target)
        assert got[0] == ref[0]
        assert got[1] == pytest.approx(ref[1], rel=1e-9, abs=1e-9)


def test_rejects_bad_curves():
    sp = _spear()
    with pytest.raises(sp.SpearError):
        sp.spear_chunk_select([([512, 256], [1.0, 2.0])], [([1], [1.0])], 1, [256], 10.0)
    with pytest.raises(sp.SpearError):
        sp.spear_chunk_select([([256], [-1.0])], [([1], [1.0])], 1, [256], 10.0)
