"""Host-side STS fitting tool ("DSpark" §3.2, STS): ECE and the left-to-right
grid search, pinned against closed forms and a synthetic head whose true
temperatures are known."""
import numpy as np
import pytest

from semi_autoregressive_speculative_gb300 import sts


def test_ece_closed_forms():
    # every prediction 1, every label 0: error 1
    assert sts.ece(np.ones(10), np.zeros(10)) == pytest.approx(1.0)
    # two bins, each calibrated on average: error 0
    p = np.array([0.1, 0.1, 0.9, 0.9, 0.9, 0.9, 0.9, 0.9, 0.9, 0.9])
    y = np.array([0, 0, 1, 1, 1, 1, 1, 1, 1, 0])
    assert sts.ece(p, y, n_bins=10) == pytest.approx(0.2 * 0.1 + 0.8 * 0.025)
    # one bin: |mean p - mean y|
    p = np.array([0.2, 0.4, 0.9])
    y = np.array([1, 0, 0])
    assert sts.ece(p, y, n_bins=1) == pytest.approx(abs(p.mean() - y.mean()))
    # bin edges: 1.0 falls in the last bin, 0.5 in the upper of two
    assert sts.ece([1.0, 0.5], [1, 1], n_bins=2) == pytest.approx(0.25)
    assert sts.ece([], []) == 0.0


def test_ece_matches_a_per_sample_loop():
    rng = np.random.default_rng(0)
    p = rng.random(500)
    y = rng.random(500) < p ** 2
    M = 7
    total = 0.0
    for b in range(M):
        sel = [i for i in range(500) if min(int(p[i] * M), M - 1) == b]
        if sel:
            total += len(sel) / 500 * abs(np.mean(p[sel]) - np.mean(y[sel]))
    assert sts.ece(p, y, n_bins=M) == pytest.approx(total, abs=1e-12)


def _synthetic_blocks(rng, N, t_true):
    """Draft blocks whose head logits z are overconfident: the true chance that
    draft j is accepted, given drafts 0..j-1 were, is sigma(z_j / t_true[j])."""
    gamma = len(t_true)
    z = rng.normal(1.5, 2.5, size=(N, gamma))
    p_true = 1.0 / (1.0 + np.exp(-z / np.asarray(t_true)[None, :]))
    ok = rng.random((N, gamma)) < p_true
    n_accept = np.where(ok.all(axis=1), gamma, np.argmin(ok, axis=1))
    return z, n_accept


def test_fit_recovers_known_temperatures():
    rng = np.random.default_rng(1)
    t_true = np.array([2.0, 1.5, 3.0, 1.0, 2.5])
    z, n_accept = _synthetic_blocks(rng, 200_000, t_true)
    t, before, after = sts.fit_sts(z, n_accept)
    assert t.dtype == np.float32 and t.shape == (5,)
    # the later positions see fewer surviving blocks, hence a looser bound
    np.testing.assert_allclose(t[:3], t_true[:3], rtol=0.08)
    np.testing.assert_allclose(t, t_true, rtol=0.25)
    assert np.all(after <= before + 1e-12)
    assert np.all(after < 0.01)
    assert before[0] > 0.03


def test_fit_keeps_a_calibrated_head_and_preserves_order():
    rng = np.random.default_rng(2)
    z, n_accept = _synthetic_blocks(rng, 100_000, [1.0, 1.0, 1.0])
    t, before, after = sts.fit_sts(z, n_accept)
    np.testing.assert_allclose(t, 1.0, rtol=0.1)
    c_raw, _ = sts.apply_sts(z, np.ones(3))
    c_fit, a_fit = sts.apply_sts(z, t)
    for j in range(3):  # the transform keeps each position's ranking
        np.testing.assert_array_equal(np.argsort(c_raw[:, j], kind="stable"),
                                      np.argsort(c_fit[:, j], kind="stable"))
    np.testing.assert_allclose(a_fit, np.cumprod(c_fit, axis=1))


def test_fit_is_sequential():
    # position 1 is fitted against a_1 = c_0(t_0) * c_1(t_1) with t_0 already
    # fixed: refitting position 1 alone from the fitted prefix gives the same t_1
    rng = np.random.default_rng(4)
    z, n_accept = _synthetic_blocks(rng, 50_000, [2.0, 0.7])
    grid = sts.default_grid(61)
    t, _, _ = sts.fit_sts(z, n_accept, grid=grid)
    prefix = 1.0 / (1.0 + np.exp(-z[:, 0] / float(t[0])))
    errs = [sts.ece(prefix / (1.0 + np.exp(-z[:, 1] / g)), n_accept > 1) for g in grid]
    assert float(t[1]) == pytest.approx(grid[int(np.argmin(errs))], rel=1e-6)


def test_logit_round_trip_and_validation():
    z = np.array([[-3.0, 0.0, 2.5]])
    c, _ = sts.apply_sts(z, np.ones(3))
    np.testing.assert_allclose(sts.logits_from_confidence(c), z, atol=1e-12)
    with pytest.raises(ValueError):
        sts.fit_sts(z, np.array([4]))
    with pytest.raises(ValueError):
        sts.fit_sts(z, np.array([1]), grid=[0.0, 1.0])
    with pytest.raises(ValueError):
        sts.apply_sts(z, np.ones(2))
