"""GPU parity of dspark_confidence and dspark_schedule against the oracle.

Confidence is fed synthetic token ids (valid inputs of any origin); the
scheduler is fed the oracle's survival products, so its outputs must match
bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import PROB_TOL, device_round, host, weights
from oracle import cost_model
from semi_autoregressive_speculative_gb300 import synth

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny_r4_g7_v4096"]


def _tokens(wl, seed=0):
    return np.random.default_rng([wl.seed, 77, seed]).integers(0, wl.V, (wl.R, wl.gamma)).astype(np.int32)


@pytest.mark.parametrize("wl", [
    TINY,
    synth.scaled(TINY, R=7, gamma=5, V=1000, d=300, name="d300_odd"),     # d not a multiple of 8
    synth.scaled(TINY, R=3, gamma=33, V=64, d=8, rank=64, name="g33"),     # gamma > warps per CTA
    synth.scaled(TINY, R=2, gamma=64, V=64, d=40, name="g64"),             # the most positions accepted
    synth.WORKLOADS["r128_g16_v151936"],
    synth.WORKLOADS["r256_g16_v129280_d7168"],
], ids=lambda w: w.name)
def test_confidence(wl):
    dr, inp = device_round(wl)
    W1, _, w = weights(wl)
    tok = _tokens(wl)
    dr.tokens.copy_(torch.from_numpy(tok))
    dr.confidence()
    c_g, a_g = host(dr.c), host(dr.a)
    c_o, a_o = oracle.confidence(inp.h, W1, w, inp.anchors, tok)
    assert np.max(np.abs(c_g - c_o)) <= PROB_TOL
    assert np.max(np.abs(a_g - a_o)) <= PROB_TOL
    assert np.all(np.diff(a_g, axis=1) <= 0)
    assert dr.status() == 0


@pytest.mark.parametrize("wl", [
    TINY,
    synth.scaled(TINY, R=3, gamma=33, V=64, d=8, rank=64, name="g33"),
    synth.WORKLOADS["r128_g16_v151936"],
], ids=lambda w: w.name)
def test_confidence_sts(wl):
    # sequential temperature scaling ("DSpark" §3.2): c_j = sigma(logit_j / t_j)
    dr, inp = device_round(wl)
    W1, _, w = weights(wl)
    tok = _tokens(wl, 1)
    t = np.random.default_rng([wl.seed, 78]).uniform(0.3, 4.0, wl.gamma).astype(np.float32)
    t[0] = 1.0
    dr.tokens.copy_(torch.from_numpy(tok))
    dr.confidence(sts_temperature=torch.from_numpy(t).cuda())
    c_g, a_g = host(dr.c), host(dr.a)
    c_o, a_o = oracle.confidence(inp.h, W1, w, inp.anchors, tok, sts_temperature=t)
    assert np.max(np.abs(c_g - c_o)) <= PROB_TOL
    assert np.max(np.abs(a_g - a_o)) <= PROB_TOL
    assert dr.status() == 0
    # unit temperatures give the unscaled head exactly
    dr.confidence(sts_temperature=torch.ones(wl.gamma, device="cuda"))
    c_1 = host(dr.c)
    dr.confidence()
    assert np.array_equal(c_1, host(dr.c))


def test_confidence_sts_bad_temperature_is_reported():
    dr, _ = device_round(TINY)
    t = torch.ones(TINY.gamma, device="cuda")
    t[2] = 0.0
    dr.confidence(sts_temperature=t)
    torch.cuda.synchronize()
    assert dr.status() & 1  # DSPARK_STATUS_NONFINITE
    with pytest.raises(ValueError):
        dr.confidence(sts_temperature=torch.ones(TINY.gamma + 1, device="cuda"))


def _schedule_both(dr, a, sps, mode, K=0):
    dr.sps[: len(sps)].copy_(torch.from_numpy(sps))
    a_dev = torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    dr.schedule(mode, K, a=a_dev)
    torch.cuda.synchronize()
    got = dict(lens=host(dr.lens)[: a.shape[0]], total_b=int(dr.sched_out[0]), argmax_b=int(dr.sched_out[1]),
               theta=float(dr.theta[0]))
    exp = oracle.schedule(a, sps, mode, K)
    return got, exp


def _assert_same(got, exp):
    assert np.array_equal(got["lens"], exp["lens"])
    assert got["total_b"] == exp["total_b"]
    assert got["argmax_b"] == exp["argmax_b"]
    assert got["theta"] == exp["theta"]  # same fp64 operations in the same order


@pytest.mark.parametrize("R,gamma,seed", [(4, 7, 0), (3, 1, 1), (1, 16, 2), (33, 5, 3), (128, 16, 4),
                                          (512, 16, 5), (8192, 1, 6), (100, 17, 7)])
def test_schedule_random(R, gamma, seed):
    from semi_autoregressive_speculative_gb300.round import DeviceRound
    rng = np.random.default_rng(seed)
    c = rng.uniform(0.3, 1.0, (R, gamma)).astype(np.float32)
    c[rng.uniform(size=c.shape) < 0.05] = 1.0   # ties inside a request
    a = oracle.survival(c)
    dr = DeviceRound(R, gamma, 64, 64, 8)
    knee = R * (1 + gamma) * rng.uniform(0.2, 0.9)
    B = np.arange(R * (1 + gamma) + 1, dtype=np.float64)
    sps = 1.0 / np.maximum(1.0, B / knee)
    for mode, K in [(0, 0), (1, 0), (1, R * gamma // 3), (1, 10**9), (2, 0)]:
        got, exp = _schedule_both(dr, a, sps, mode, K)
        _assert_same(got, exp)


@pytest.mark.parametrize("R,gamma,seed", [(4, 7, 10), (33, 5, 11), (128, 16, 12), (512, 16, 13), (100, 17, 14)])
def test_schedule_rows_that_rise(R, gamma, seed):
    """a that is not a survival product (it rises along some requests, and
    has ties across requests): the kernel's general sort path, against the
    oracle."""
    from semi_autoregressive_speculative_gb300.round import DeviceRound
    rng = np.random.default_rng(seed)
    a = rng.uniform(0.0, 1.0, (R, gamma)).astype(np.float32)
    a[rng.uniform(size=a.shape) < 0.05] = 0.5   # ties inside and across requests
    dr = DeviceRound(R, gamma, 64, 64, 8)
    knee = R * (1 + gamma) * rng.uniform(0.2, 0.9)
    B = np.arange(R * (1 + gamma) + 1, dtype=np.float64)
    sps = 1.0 / np.maximum(1.0, B / knee)
    for mode, K in [(0, 0), (1, R * gamma // 3), (2, 0)]:
        got, exp = _schedule_both(dr, a, sps, mode, K)
        _assert_same(got, exp)


@pytest.mark.parametrize("case", ["zeros_and_halves", "large_values"])
def test_schedule_edge_values(case):
    """Values that exercise the fixed-point and Theta arithmetic, against the
    oracle bit for bit: signed zeros (-0 ties with 0, broken by (j, r)),
    subnormals (round to 0 in Q.40), values whose Q.40 image is an exact half
    (ties to even), and a above 1 (not survival products, but admissible) large
    enough that R + S_b no longer fits 53 bits."""
    from semi_autoregressive_speculative_gb300.round import DeviceRound
    rng = np.random.default_rng(21)
    R, gamma = 33, 7
    if case == "zeros_and_halves":
        # descending; in Q.40: 1.5 -> 2, 1.25 -> 1, 0.5 -> 0, 0.25 -> 0, a subnormal -> 0
        pool = np.array([0.75, 0.5, 3 * 2.0 ** -41, 5 * 2.0 ** -42, 2.0 ** -41, 2.0 ** -42, 1e-45, 0.0, -0.0],
                        dtype=np.float32)
        # each request a non-increasing run drawn from the pool (-0 and 0 compare equal)
        a = np.stack([pool[np.sort(rng.integers(0, len(pool), gamma))] for _ in range(R)])
    else:
        a = np.sort(rng.uniform(1.0, 4.0e6, (R, gamma)), axis=1)[:, ::-1].astype(np.float32)
        assert float(a.astype(np.float64).sum()) > 2.0 ** 13  # R 2^40 + S_n above 2^53
    dr = DeviceRound(R, gamma, 64, 64, 8)
    B = np.arange(R * (1 + gamma) + 1, dtype=np.float64)
    sps = 1.0 / np.maximum(1.0, B / (R * 3.0))
    for mode, K in [(0, 0), (1, R * gamma // 2), (2, 0)]:
        got, exp = _schedule_both(dr, a, sps, mode, K)
        _assert_same(got, exp)


def test_schedule_handbook_planner_inputs():
    # the page's adaptive-planner confidences, batch 512 x 7, against the oracle
    torch_ = pytest.importorskip("torch")
    torch_.manual_seed(0)
    from semi_autoregressive_speculative_gb300.round import DeviceRound
    K = 7
    for batch in (16, 128, 512):
        good = batch // 2
        level = torch_.cat([torch_.full((good, K), 0.9), torch_.full((batch - good, K), 0.55)])
        conf = (level * torch_.rand(batch, K).mul(0.2).add(0.9)).clamp(max=0.99).numpy()
        a = oracle.survival(conf)
        sps = np.array([cost_model.sps_with_draft(B) for B in range(batch * (1 + K) + 1)])
        dr = DeviceRound(batch, K, 64, 64, 8)
        got, exp = _schedule_both(dr, a, sps, 0)
        _assert_same(got, exp)
        assert got["total_b"] == {16: 112, 128: 57, 512: 7}[batch]


def test_schedule_staircase_full_size_and_lag():
    wl = synth.WORKLOADS["r512_g16_v32768_staircase"]
    from semi_autoregressive_speculative_gb300.round import DeviceRound
    dr = DeviceRound(wl.R, wl.gamma, 64, 64, 8)
    sps = synth.sps_table(wl)
    W1, _, w = weights(wl)
    history = []
    for rnd in range(wl.rounds):
        inp = synth.round_inputs(wl, rnd)
        tok = np.random.default_rng([wl.seed, 78, rnd]).integers(0, wl.V, (wl.R, wl.gamma)).astype(np.int32)
        _, a = oracle.confidence(inp.h, W1, w, inp.anchors, tok)
        for mode in (0, 1):
            K = wl.R * wl.gamma if len(history) < 2 else history[-2]
            got, exp = _schedule_both(dr, a, sps, mode, K)
            _assert_same(got, exp)
        history.append(exp["argmax_b"])
