"""Pins of the oracle's hardware-aware prefix scheduler ("DSpark" page §4.1-4.3;
"DSpark: Speculative decodingを活用したLLM推論の高速化" page, "スケジューラの実運用適用").

Brute force: for tiny R and gamma, every verify-length vector l in
{0..gamma}^R is scored directly as Theta = (sum_r 1 + sum_{j<=l_r} a_rj) * SPS(B),
B = sum_r (1 + l_r), in fp64 without sorting.  The global optimum must equal
the best budget on the oracle's sorted path, the admitted sets must be
per-request prefixes, and early stop must reach the optimum whenever Theta
is unimodal along the path.
"""
import itertools

import numpy as np

from semi_autoregressive_speculative_gb300 import synth


def _survival(rng, R, gamma, orc):
    c = rng.uniform(0.2, 1.0, (R, gamma)).astype(np.float32)
    return orc.survival(c)


def _brute(a, sps):
    R, gamma = a.shape
    best, best_l = -1.0, None
    a64 = a.astype(np.float64)
    for ls in itertools.product(range(gamma + 1), repeat=R):
        tau = sum(1.0 + a64[r, :l].sum() for r, l in enumerate(ls))
        th = tau * sps[R + sum(ls)]
        if th > best:
            best, best_l = th, ls
    return best, best_l


def _knee_sps(n, knee):
    B = np.arange(n + 1, dtype=np.float64)
    return 1.0 / np.maximum(1.0, B / knee)


def test_exhaustive_small_cases(orc):
    rng = np.random.default_rng(0)
    checked_unimodal = 0
    for trial in range(60):
        R = int(rng.integers(1, 4))
        gamma = int(rng.integers(1, 4))
        a = _survival(rng, R, gamma, orc)
        knee = float(rng.uniform(R, R * (1 + gamma) + 1))
        sps = _knee_sps(R * (1 + gamma), knee)
        best, best_l = _brute(a, sps)
        res = orc.schedule(a, sps, orc.MODE_TOP_K, 10**6)  # any mode gives argmax_b and theta_all
        th = res["theta_all"]
        assert abs(th[res["argmax_b"]] - best) <= 1e-9 * best
        # sets on the sorted path are per-request prefixes
        for b in range(R * gamma + 1):
            r_b = orc.schedule(a, sps, orc.MODE_TOP_K, b)
            lens = r_b["lens"]
            assert lens.sum() == b and r_b["total_b"] == b
            admitted = [(r, j) for r in range(R) for j in range(lens[r])]
            tau = sum(1.0 + a[r, :lens[r]].astype(np.float64).sum() for r in range(R))
            assert abs(tau * sps[R + b] - th[b]) <= 1e-9 * th[b]
            assert len(admitted) == b
        # early stop reaches the optimum when Theta is unimodal on the path
        d = np.diff(th)
        unimodal = not np.any((d[1:] > 0) & (d[:-1] <= 0))
        es = orc.schedule(a, sps, orc.MODE_EARLY_STOP)
        if unimodal:
            checked_unimodal += 1
            assert abs(es["theta"] - best) <= 1e-9 * best
    assert checked_unimodal > 20


def test_early_stop_is_first_non_improvement(orc):
    a = np.array([[0.9, 0.5, 0.1], [0.8, 0.8, 0.7]], np.float32)
    sps = np.ones(2 * 4 + 1)
    sps[4:] = 0.5  # a cliff at B = 4 (b = 2)
    res = orc.schedule(a, sps, orc.MODE_EARLY_STOP)
    # path: 0.9, 0.8, 0.8, 0.7, 0.5, 0.1 -> Theta(1) > Theta(0), Theta(2) < Theta(1)
    assert res["total_b"] == 1
    assert res["lens"].tolist() == [1, 0]
    # a tie counts as a drop (admit only on strict improvement)
    a2 = np.array([[0.0, 0.0]], np.float32)
    res2 = orc.schedule(a2, np.ones(4), orc.MODE_EARLY_STOP)
    assert res2["total_b"] == 0 and res2["argmax_b"] == 0


def test_sort_ties_keep_prefixes(orc):
    # c = 1 makes a tie within a request; position order must keep prefixes
    a = np.array([[1.0, 1.0, 1.0], [1.0, 0.5, 0.5]], np.float32)
    sps = np.ones(2 * 4 + 1)
    for b in range(7):
        lens = orc.schedule(a, sps, orc.MODE_TOP_K, b)["lens"]
        # (a desc, j asc, r asc): (r0,j0) (r1,j0) (r0,j1) (r0,j2) (r1,j1) (r1,j2)
        expect = [[0, 0], [1, 0], [1, 1], [2, 1], [3, 1], [3, 2], [3, 3]][b]
        assert lens.tolist() == expect


def test_modes(orc):
    rng = np.random.default_rng(1)
    a = _survival(rng, 5, 4, orc)
    sps = _knee_sps(5 * 5, 9.0)
    fixed = orc.schedule(a, sps, orc.MODE_FIXED)
    assert fixed["total_b"] == 20 and fixed["lens"].tolist() == [4] * 5
    assert orc.schedule(a, sps, orc.MODE_TOP_K, 999)["total_b"] == 20
    assert orc.schedule(a, sps, orc.MODE_TOP_K, -3)["total_b"] == 0
    assert orc.schedule(a, sps, orc.MODE_TOP_K, 7)["total_b"] == 7


def test_staircase_early_stop_vs_lagged_top_k(orc):
    # The staircase SPS table of the R=512 workload has cliffs at B = 1024,
    # 2048, 4096, so Theta is not unimodal: early stop halts at the first
    # cliff while the global optimum lies beyond it.  Top-K with K equal to
    # the global argmax reaches the optimum ("DSpark" page §4.2-4.3).
    wl = synth.WORKLOADS["r512_g16_v32768_staircase"]
    rng = np.random.default_rng(3)
    R, gamma = wl.R, wl.gamma
    c = np.empty((R, gamma), np.float32)
    c[: R // 2] = rng.uniform(0.9, 0.99, (R // 2, gamma))
    c[R // 2:] = rng.uniform(0.3, 0.6, (R - R // 2, gamma))
    a = orc.survival(c)
    sps = synth.sps_table(wl)
    es = orc.schedule(a, sps, orc.MODE_EARLY_STOP)
    assert es["total_b"] == 1024 - R - 1  # B = R + b stays just below the cliff at 1024
    best = es["argmax_b"]
    th = es["theta_all"]
    assert th[best] > es["theta"] * 1.05
    tk = orc.schedule(a, sps, orc.MODE_TOP_K, best)
    assert tk["total_b"] == best and abs(tk["theta"] - th.max()) == 0.0
