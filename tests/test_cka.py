"""Linear CKA (Technical Summary 2.1 B: the training-free damage proxy that
feeds module selection), host: spear_linear_cka against the oracle's HSIC
definition, its invariances and a closed form; damage scores drive the
selection rule."""
import numpy as np
import pytest

import oracle


def _spear():
    from quantized_gemm_error_gb300 import spear
    spear.load()
    return spear


@pytest.mark.parametrize("n,dx,dy", [(40, 64, 48), (200, 16, 24), (33, 33, 7)])   # token- and feature-space forms
def test_matches_the_hsic_definition(n, dx, dy):
    rng = np.random.default_rng(n + dx)
    X = rng.standard_normal((n, dx)).astype(np.float32)
    Y = (X[:, :min(dx, dy)] @ rng.standard_normal((min(dx, dy), dy)) * 0.3
         + rng.standard_normal((n, dy))).astype(np.float32)
    got = _spear().spear_linear_cka(X, Y)
    assert got == pytest.approx(oracle.linear_cka(X, Y), rel=1e-9, abs=1e-12)
    assert 0.0 <= got <= 1.0


def test_identity_symmetry_and_invariances():
    sp = _spear()
    rng = np.random.default_rng(3)
    X = rng.standard_normal((96, 40)).astype(np.float32)
    Y = (X @ rng.standard_normal((40, 30)) + 2 * rng.standard_normal((96, 30))).astype(np.float32)
    base = sp.spear_linear_cka(X, Y)
    assert sp.spear_linear_cka(X, X) == pytest.approx(1.0, abs=1e-12)
    assert sp.spear_linear_cka(Y, X) == pytest.approx(base, rel=1e-12)
    Q, _ = np.linalg.qr(rng.standard_normal((40, 40)))
    assert sp.spear_linear_cka((X @ Q).astype(np.float32), Y) == pytest.approx(base, rel=1e-6)   # orthogonal
    assert sp.spear_linear_cka(X * np.float32(7.5), Y) == pytest.approx(base, rel=1e-6)          # isotropic scale
    assert sp.spear_linear_cka(X + np.float32(3.0), Y) == pytest.approx(base, rel=1e-6)          # mean shift


def test_rank_one_is_the_squared_correlation():
    rng = np.random.default_rng(4)
    a = rng.standard_normal(500)
    b = 0.6 * a + rng.standard_normal(500)
    got = _spear().spear_linear_cka(a[:, None].astype(np.float32), b[:, None].astype(np.float32))
    r = np.corrcoef(a.astype(np.float32), b.astype(np.float32))[0, 1]
    assert got == pytest.approx(r * r, rel=1e-6)


def test_damage_scores_select_the_damaged_modules():
    """Four modules whose 'quantised' outputs carry growing noise: the two
    noisiest get the compensators."""
    sp = _spear()
    rng = np.random.default_rng(5)
    ref, quant = [], []
    for noise in (0.01, 0.02, 1.0, 1.5):
        R = rng.standard_normal((128, 64)).astype(np.float32)
        ref.append(R)
        quant.append((R + noise * rng.standard_normal(R.shape)).astype(np.float32))
    dmg = sp.cka_damage(ref, quant)
    assert np.all(np.diff(dmg) > 0)
    mask, ranks = sp.spear_layer_select_mask(dmg, np.ones(4, np.float32), 64.0, 16, 32)
    assert mask.tolist() == [0, 0, 1, 1] and set(ranks[2:].tolist()) == {32}


def test_damage_score_is_one_minus_cka_computed_by_the_library():
    """spear_cka_damage (C ABI) equals 1 - spear_linear_cka on the same inputs,
    and is checked the same way."""
    sp = _spear()
    rng = np.random.default_rng(9)
    X = rng.standard_normal((96, 40)).astype(np.float32)
    Y = (X[:, :24] + 0.3 * rng.standard_normal((96, 24))).astype(np.float32)
    assert sp.spear_cka_damage(X, Y) == 1.0 - sp.spear_linear_cka(X, Y)
    assert sp.spear_cka_damage(X, X) == pytest.approx(0.0, abs=1e-12)
    with pytest.raises(sp.SpearError):
        sp.spear_cka_damage(np.ones((10, 4), np.float32), X[:10])


def test_rejects_degenerate_inputs():
    sp = _spear()
    X = np.ones((10, 4), np.float32)
    with pytest.raises(sp.SpearError):
        sp.spear_linear_cka(X, np.random.default_rng(0).standard_normal((10, 3)).astype(np.float32))   # no variance
    with pytest.raises(sp.SpearError):
        sp.spear_linear_cka(np.array([[1.0, np.nan], [0.0, 1.0]], np.float32), np.eye(2, dtype=np.float32))
