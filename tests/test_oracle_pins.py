"""Pins for the CPU oracle (no GPU): each test checks the oracle against
something other than itself -- a library routine, a closed form, an invariant
the definition fixes, or a hand-worked example (tests/golden/).

Source of the method: the SPEAR explainer (gist.science), Technical Summary
2.1 A (effective weight W + alpha*B*diag(gate)*A, input-adaptive gate),
2.1 B (entropy-aware module selection), 3.1 (RTN per-channel int4).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from quantized_gemm_error_gb300.inputs import (bf16_bits_to_f32, f32_to_bf16_bits, make_layer,
                                               make_tokens)

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


# ----------------------------------------------------------------- numbers

def _f16_ru_reference(v: np.float32) -> int:
    """Smallest binary16 value >= v, via numpy's own float16 (round to nearest)."""
    with np.errstate(over="ignore"):
        h = np.float16(v)
        if np.isnan(h):
            return 0x7E00
        if np.float32(h) < v:
            h = np.nextafter(h, np.float16(np.inf), dtype=np.float16)
    return int(np.array(h, dtype=np.float16).view(np.uint16))


def test_f16_ru_matches_numpy_definition():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(0.01),
        rng.standard_normal(2000).astype(np.float32) * np.float32(1000.0),
        (rng.random(2000).astype(np.float32) * np.float32(1e-6)),           # fp16 subnormals
        np.array([0.0, -0.0, 65504.0, 65505.0, 65519.0, 65520.0, 70000.0, -65504.0, -65505.0,
                  -70000.0, 2.0 ** -24, 2.0 ** -25, 3e-8, -3e-8, 2.0 ** -14, 1e-40, -1e-40],
                 dtype=np.float32),
    ])
    for v in vals:
        got = oracle.f32_to_f16_ru(float(v))
        ref = _f16_ru_reference(np.float32(v))
        if np.float32(v) == 0.0:
            assert got & 0x7FFF == 0
        else:
            assert got == ref, (float(v), hex(got), hex(ref))


def test_f16_to_f32_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_to_f32(int(b)) for b in bits], dtype=np.float32)
    same = (got.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_bf16_rn_matches_torch():
    rng = np.random.default_rng(2)
    vals = np.concatenate([rng.standard_normal(5000).astype(np.float32) * 37.0,
                           np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0, 3e38],
                                    dtype=np.float32)])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16_rn(float(v)) for v in vals], dtype=np.uint16)
    assert (got == ref).all()
    # and the input generator's cast agrees with torch too (both sides read it)
    assert (f32_to_bf16_bits(vals) == ref).all()


# --------------------------------------------------------------- quantiser

@pytest.mark.parametrize("case", ["pack_sym_per_channel", "pack_asym_group"])
def test_pack_worked_example(case):
    ex = GOLDEN[case]
    W = np.array([ex["W_row"]], dtype=np.float32)
    q, s, z = oracle.quantize_pack(W, ex["G"], ex["sym"])
    assert list(q[0]) == ex["bytes"]
    assert int(s[0, 0]) == ex["scale_bits"]
    assert list(oracle.unpack_codes(q, W.shape[1])[0]) == ex["codes"]
    if not ex["sym"]:
        assert list(z[0]) == ex["zero_bytes"]


def _pack_layout_reference(codes: np.ndarray) -> np.ndarray:
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


@pytest.mark.parametrize("sym,G", [(True, None), (True, 128), (False, 128), (False, None)])
def test_pack_layout_and_error_bound(sym, G):
    """Nibble order (low nibble = even k), codes in range, |w - dq| <= s/2."""
    lay, _ = make_layer(48, 512, 0, seed=3)
    W = lay.W
    W[5, :] = 0.0                                   # an all-zero row
    W[7, 100:140] *= 40.0                           # a wide group
    K = W.shape[1]
    g = K if G is None else G
    q, s, z = oracle.quantize_pack(W, g, sym)
    codes = oracle.unpack_codes(q, K)
    assert codes.max() <= 15
    assert (_pack_layout_reference(codes) == q).all()
    dq = oracle.dequant(q, s, z, K, g, sym)
    svals = s.view(np.float16).astype(np.float64)
    s_full = np.repeat(svals, g, axis=1)
    err = np.abs(W.astype(np.float64) - dq)
    assert (err <= s_full * (0.5 + 2.0 ** -20)).all()
    # the scale is the fp16 value just at or above the exact fp32 ratio
    zq = oracle.unpack_zeros(z, W.shape[0], K, g, sym)
    for n in (0, 7, 19):
        for gi in range(K // g):
            w = W[n, gi * g:(gi + 1) * g]
            if sym:
                s32 = np.float32(np.abs(w).max()) / np.float32(7.0)
            else:
                s32 = (np.float32(max(w.max(), 0)) - np.float32(min(w.min(), 0))) / np.float32(15.0)
            sv = np.float16(svals[n, gi])
            assert np.float32(sv) >= s32
            below = np.nextafter(sv, np.float16(-np.inf), dtype=np.float16)
            assert s32 == 0 or np.float32(below) < s32
            c = codes[n, gi * g:(gi + 1) * g].astype(int) - int(zq[n, gi])
            if sym:
                assert np.abs(c).max() == 7           # amax maps onto +-7
            else:
                assert c[np.argmin(w)] + zq[n, gi] == 0 or w.min() >= 0   # min maps onto code 0
    assert (codes[5] == (8 if sym else 0)).all() and (svals[5] == 0).all()


@pytest.mark.parametrize("sym", [True, False])
def test_pack_exact_grid_round_trips(sym):
    """Weights that already lie on an fp16-scaled int grid come back unchanged."""
    rng = np.random.default_rng(4)
    N, K, G = 16, 256, 64
    s = np.float16(rng.uniform(0.01, 0.2, size=(N, K // G))).astype(np.float32)
    if sym:
        q = rng.integers(-7, 8, size=(N, K))
        q[:, ::G] = 7                               # +-7 present in every group
        q[:, 1::G] = -7
        W = (q * np.repeat(s, G, axis=1)).astype(np.float32)
    else:
        u = rng.integers(0, 16, size=(N, K))
        u[:, ::G] = 0
        u[:, 1::G] = 15
        z = rng.integers(0, 16, size=(N, K // G))
        W = ((u - np.repeat(z, G, axis=1)) * np.repeat(s, G, axis=1)).astype(np.float32)
    qw, sc, zz = oracle.quantize_pack(W, G, sym)
    dq = oracle.dequant(qw, sc, zz, K, G, sym)
    assert (dq == W.astype(np.float64)).all()
    assert (sc.view(np.float16).astype(np.float32) == s).all()


def test_pack_rejects_non_finite_and_overflow():
    W = np.zeros((2, 8), np.float32)
    W[1, 3] = np.nan
    with pytest.raises(ValueError):
        oracle.quantize_pack(W, 8, True)
    W[1, 3] = 1e9                                    # 1e9/7 overflows fp16
    with pytest.raises(ValueError):
        oracle.quantize_pack(W, 8, True)


# ------------------------------------------------------------------- layer

def _layer_dict(lay, G, sym, comp=True, b_g=None):
    q, s, z = oracle.quantize_pack(lay.W, G, sym)
    return dict(N=lay.N, K=lay.K, G=G, sym=sym, qweight=q, scales=s, zeros=z, r=lay.r, A=lay.A,
                B=lay.B, w_g=lay.w_g, b_g=lay.b_g if b_g is None else b_g, alpha=lay.alpha,
                comp_enabled=int(comp))


def test_linear_worked_example():
    ex = GOLDEN["linear_tiny"]
    W = np.array(ex["W"], np.float32)
    x = f32_to_bf16_bits(np.array(ex["x"], np.float32))
    q, s, z = oracle.quantize_pack(W, ex["G"], ex["sym"])
    assert oracle.unpack_codes(q, ex["K"]).tolist() == ex["codes"]
    assert list(s.view(np.float16).astype(np.float64)[:, 0]) == ex["scale_values"]
    for case in ex["cases"]:
        L = dict(N=2, K=4, G=4, sym=True, qweight=q, scales=s, zeros=None, r=2,
                 A=f32_to_bf16_bits(np.array(ex["A"], np.float32)),
                 B=f32_to_bf16_bits(np.array(ex["B"], np.float32)),
                 w_g=f32_to_bf16_bits(np.array(case["w_g"], np.float32)),
                 b_g=case["b_g"], alpha=ex["alpha"], comp_enabled=1)
        y, corr, gate = oracle.linear(L, x, want_corr=True, want_gate=True)
        assert gate[0] == pytest.approx(case["gate"], abs=1e-15)
        np.testing.assert_allclose(y, np.array(case["y"]), rtol=0, atol=1e-12)
        np.testing.assert_allclose(y - corr, np.array(ex["y_main"]), rtol=0, atol=0)


@pytest.mark.parametrize("sym,G", [(True, 256), (False, 64)])
def test_main_term_is_the_textbook_matmul(sym, G):
    lay, rng = make_layer(40, 256, 8, seed=5)
    x = make_tokens(rng, 5, 256, outlier_frac=0.02)
    L = _layer_dict(lay, G, sym, comp=False)
    y = oracle.linear(L, x)
    dq = oracle.dequant(L["qweight"], L["scales"], L["zeros"], 256, G, sym)
    ref = bf16_bits_to_f32(x).astype(np.float64) @ dq.T            # numpy matmul
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_gate_closed_forms_and_identities():
    lay, rng = make_layer(32, 128, 16, seed=6)
    x = make_tokens(rng, 4, 128)
    xf = bf16_bits_to_f32(x).astype(np.float64)
    Af = bf16_bits_to_f32(lay.A).astype(np.float64)
    Bf = bf16_bits_to_f32(lay.B).astype(np.float64)
    base = _layer_dict(lay, 128, True)
    # gate forced to 0 (b_g -> -inf) gives exactly the plain W4 output
    y, corr, gate = oracle.linear({**base, "b_g": -1e30}, x, want_corr=True, want_gate=True)
    assert (gate == 0).all() and (corr == 0).all()
    assert (y == oracle.linear({**base, "comp_enabled": 0}, x)).all()
    # rank 0 and B = 0 give the plain output too
    assert (oracle.linear({**base, "r": 0, "A": None, "B": None}, x) == y).all()
    assert (oracle.linear({**base, "B": np.zeros_like(lay.B)}, x) == y).all()
    # w_g = 0, b_g = 0: gate is exactly 1/2, correction = 0.5 * B (A x)
    y5, c5, g5 = oracle.linear({**base, "w_g": np.zeros_like(lay.w_g), "b_g": 0.0}, x,
                               want_corr=True, want_gate=True)
    assert (g5 == 0.5).all()
    np.testing.assert_allclose(c5, 0.5 * (xf @ Af.T) @ Bf.T, rtol=1e-12, atol=1e-15)
    # w_g = e_7: the gate reads channel 7 of the token, sigmoid(x[m, 7] + b_g)
    e7 = np.zeros(128, np.float32); e7[7] = 1.0
    _, c7, g7 = oracle.linear({**base, "w_g": f32_to_bf16_bits(e7), "b_g": 0.25}, x,
                              want_corr=True, want_gate=True)
    sig = 1.0 / (1.0 + np.exp(-(xf[:, 7] + 0.25)))
    np.testing.assert_allclose(g7, sig, rtol=1e-14)
    np.testing.assert_allclose(c7, sig[:, None] * ((xf @ Af.T) @ Bf.T), rtol=1e-12, atol=1e-15)
    # linear in B and in alpha
    B2 = f32_to_bf16_bits(2.0 * bf16_bits_to_f32(lay.B))
    _, c2, _ = oracle.linear({**base, "B": B2}, x, want_corr=True)
    _, c1, _ = oracle.linear(base, x, want_corr=True)
    np.testing.assert_allclose(c2, 2.0 * c1, rtol=1e-14, atol=0)
    _, c3, _ = oracle.linear({**base, "alpha": 3.0}, x, want_corr=True)
    np.testing.assert_allclose(c3, 3.0 * c1, rtol=1e-14, atol=0)


def test_tokens_are_independent_and_columns_selectable():
    lay, rng = make_layer(24, 256, 16, seed=7)
    x = make_tokens(rng, 6, 256, outlier_frac=0.05)
    L = _layer_dict(lay, 128, False)
    y = oracle.linear(L, x)
    perm = np.array([3, 0, 5, 1, 4, 2])
    assert (oracle.linear(L, x[perm]) == y[perm]).all()
    idx = np.array([23, 0, 11, 11])
    assert (oracle.linear(L, x, n_idx=idx) == y[:, idx]).all()
    assert (oracle.linear(L, x, nthreads=4) == y).all()
    assert oracle.linear(L, x[:0]).shape == (0, 24)


def test_fp32_accumulation_within_error_bound():
    lay, rng = make_layer(16, 2048, 16, seed=8)
    x = make_tokens(rng, 3, 2048, outlier_frac=0.01)
    L = _layer_dict(lay, 128, False)
    y64, c64, _ = oracle.linear(L, x, want_corr=True)
    y32, c32, _ = oracle.linear(L, x, accum_double=False, want_corr=True)
    dq = oracle.dequant(L["qweight"], L["scales"], L["zeros"], 2048, 128, False)
    xf = bf16_bits_to_f32(x).astype(np.float64)
    bound = 2048 * 2.0 ** -24 * (np.abs(xf) @ np.abs(dq).T)
    assert (np.abs((y32 - c32) - (y64 - c64)) <= bound).all()
    assert np.abs(c32 - c64).max() <= 1e-5 * np.abs(c64).max()


def test_vector_gate_reduces_to_closed_forms():
    lay, rng = make_layer(20, 128, 8, seed=9)
    x = make_tokens(rng, 3, 128)
    L = _layer_dict(lay, 64, True)
    xf = bf16_bits_to_f32(x).astype(np.float64)
    Af = bf16_bits_to_f32(lay.A).astype(np.float64)
    Bf = bf16_bits_to_f32(lay.B).astype(np.float64)
    h = 4
    zeros = lambda *s: np.zeros(s, np.float32)
    # all-zero MLP: gamma = 1/2 everywhere, matches the scalar gate at w_g = 0, b_g = 0
    y, gam = oracle.linear_vector_gate(L, x, zeros(h, 8), zeros(h), zeros(8, h), zeros(8))
    assert (gam == 0.5).all()
    ys = oracle.linear({**L, "w_g": np.zeros_like(lay.w_g), "b_g": 0.0}, x)
    np.testing.assert_allclose(y, ys, rtol=1e-13, atol=1e-15)
    # W2 = 0: gamma_j = sigmoid(c2_j), correction = B diag(gamma) A x
    c2 = np.linspace(-2, 2, 8).astype(np.float32)
    y2, gam2 = oracle.linear_vector_gate(L, x, zeros(h, 8), zeros(h), zeros(8, h), c2)
    sig = 1.0 / (1.0 + np.exp(-c2.astype(np.float64)))
    assert np.allclose(gam2, sig[None, :], rtol=1e-14)
    y_plain = oracle.linear({**L, "comp_enabled": 0}, x)
    np.testing.assert_allclose(y2 - y_plain, ((xf @ Af.T) * sig[None, :]) @ Bf.T, rtol=1e-10,
                               atol=1e-14)



def test_vector_gate_routes_single_components():
    """Sparse W1, W2 that route one rank component through one hidden unit each
    give gamma in closed form from t = A x (a textbook matmul): a transposed W1
    or W2, a dropped c1, c2 or relu changes which components move, or how."""
    lay, rng = make_layer(24, 256, 8, seed=11)
    x = make_tokens(rng, 32, 256)
    L = _layer_dict(lay, 128, False)
    t = bf16_bits_to_f32(x).astype(np.float64) @ bf16_bits_to_f32(lay.A).astype(np.float64).T   # [M][8]
    W1 = np.zeros((2, 8), np.float32)
    W1[0, 3] = 1.0                       # hidden 0 = relu(t_3 + 0.05)
    W1[1, 5] = -1.0                      # hidden 1 = relu(-t_5 - 0.02)
    c1 = np.array([0.05, -0.02], np.float32)
    W2 = np.zeros((8, 2), np.float32)
    W2[6, 0] = 8.0                       # gamma_6 = sigmoid(8 hidden_0 + c2_6)
    W2[1, 1] = -6.0                      # gamma_1 = sigmoid(-6 hidden_1 + c2_1)
    c2 = np.linspace(-1.5, 1.5, 8).astype(np.float32)
    _, gam = oracle.linear_vector_gate(L, x, W1, c1, W2, c2)
    sig = lambda v: 1.0 / (1.0 + np.exp(-v))
    h0 = np.maximum(t[:, 3] + float(c1[0]), 0.0)
    h1 = np.maximum(-t[:, 5] + float(c1[1]), 0.0)
    want = np.tile(sig(c2.astype(np.float64)), (x.shape[0], 1))
    want[:, 6] = sig(8.0 * h0 + float(c2[6]))
    want[:, 1] = sig(-6.0 * h1 + float(c2[1]))
    # both sides of each relu occur among the tokens
    assert (h0 > 0).any() and (h0 == 0).any()
    assert (h1 > 0).any() and (h1 == 0).any()
    np.testing.assert_allclose(gam, want, rtol=1e-6, atol=0)


# -------------------------------------------------------- module selection

def test_layer_select_worked_example():
    ex = GOLDEN["layer_select"]
    for case in ex["cases"]:
        m, r = oracle.layer_select_mask(ex["damage"], ex["cost"], case["budget"], case["rank_min"],
                                        case["rank_max"])
        assert m.tolist() == case["mask"] and r.tolist() == case["rank"]


def test_layer_select_invariants():
    L = 12
    cost = np.full(L, 1000.0)
    onehot = np.zeros(L); onehot[5] = 3.0
    m, r = oracle.layer_select_mask(onehot, cost, 1e6, 16, 64)
    assert m.tolist() == [0] * 5 + [1] + [0] * 6 and r[5] == 64      # concentrated -> 1 module
    m, r = oracle.layer_select_mask(np.ones(L), cost, 1e6, 16, 64)
    assert m.all() and (r == 64).all()                              # diffuse -> all modules
    rng = np.random.default_rng(10)
    d = rng.random(L) ** 3
    c = rng.uniform(500, 4000, L)
    prev = None
    for budget in np.geomspace(1e3, 1e7, 25):
        m, r = oracle.layer_select_mask(d, c, budget, 16, 128)
        used = (r * c * m).sum()
        assert used <= budget + 1e-6
        assert (r % 16 == 0).all() and ((r == 0) == (m == 0)).all()
        if prev is not None and m.sum() == prev[0].sum():
            assert r.max() >= prev[1].max()                         # more budget, rank never drops
        prev = (m, r)
    m1, r1 = oracle.layer_select_mask(d, c, 5e4, 16, 128)
    m2, r2 = oracle.layer_select_mask(d, c, 5e4, 16, 128)
    assert (m1 == m2).all() and (r1 == r2).all()
    # no damage: nothing selected
    m, r = oracle.layer_select_mask(np.zeros(L), cost, 1e6, 16, 64)
    assert not m.any()
