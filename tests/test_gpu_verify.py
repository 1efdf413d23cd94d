"""GPU parity of dspark_verify against the oracle.  Draft outputs fed to
verify come from the oracle (compared requests) or stand-ins (the rest)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (check_verify, device_round, host, oracle_confidence, oracle_draft, sample_requests,
                         verify_inputs, weights)
from semi_autoregressive_speculative_gb300 import synth
from semi_autoregressive_speculative_gb300.round import MODE_EARLY_STOP, MODE_TOP_K

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny_r4_g7_v4096"]


def _run(wl, temperature, compare, lens=None, rnd=0):
    dr, inp = device_round(wl)
    tokens, pd, lz, T, lens = verify_inputs(wl, inp, rnd, compare, temperature, lens)
    dr.T.copy_(torch.from_numpy(T))
    dr.tokens.copy_(torch.from_numpy(tokens))
    dr.pd.copy_(torch.from_numpy(pd))
    dr.logZ.copy_(torch.from_numpy(lz))
    dr.lens.copy_(torch.from_numpy(lens))
    dr.verify(temperature, wl.seed, rnd)
    na, nx = host(dr.n_accept), host(dr.next_token)
    assert np.all(na >= 0) and np.all(na <= lens)
    assert nx.min() >= 0 and nx.max() < wl.V
    ex = check_verify(wl, inp, T, tokens, lens, na, nx, temperature, rnd, compare)
    assert dr.status() == 0
    return na, nx, ex


@pytest.mark.parametrize("temperature", [1.0, 0.7, 0.0])
def test_verify_tiny(temperature):
    wl = TINY
    na, nx, ex = _run(wl, temperature, range(wl.R))
    assert ex <= 1


@pytest.mark.parametrize("temperature", [1.0, 0.0])
def test_verify_ragged_lengths(temperature):
    wl = synth.scaled(TINY, R=9, gamma=5, V=1000, d=16, name="ragged_verify")
    lens = np.array([0, 1, 2, 3, 4, 5, 5, 0, 2], np.int32)
    na, nx, ex = _run(wl, temperature, range(wl.R), lens=lens)
    assert ex <= 1


@pytest.mark.parametrize("temperature", [1.0, 0.0])
def test_verify_max_positions(temperature):
    # gamma = 64, the most positions the boundary accepts, lengths from 0 to 64
    wl = synth.scaled(TINY, R=5, gamma=64, V=1000, d=16, name="verify_g64")
    lens = np.array([0, 1, 31, 63, 64], np.int32)
    na, nx, ex = _run(wl, temperature, range(wl.R), lens=lens)
    assert ex <= 1


def test_verify_many_rows_two_mtiles():
    wl = synth.scaled(TINY, R=140, gamma=3, V=2048, rank=128, d=16, name="verify_r140")
    na, nx, ex = _run(wl, 1.0, range(0, 140, 7))
    assert ex <= 1


@pytest.mark.parametrize("name", ["r32_g7_v151936", "r256_g16_v129280_d7168"])
def test_verify_full_size_sampled(name):
    wl = synth.WORKLOADS[name]
    for temperature in wl.temperatures:
        rows = sample_requests(wl.R)
        na, nx, ex = _run(wl, temperature, rows)
        assert ex <= max(1, len(rows) // 4)  # each exemption checked within tolerance


def test_verify_full_size_staircase_every_request():
    # The scheduler/verify stress workload at full size (R = 512: four
    # M-tiles; V = 32768; target noise std 0.3 on the first half of the
    # requests, 2 on the second), every request compared with the oracle.
    # Draft, confidence and both schedules come from the oracle on all
    # requests, so that verify sees the ragged lengths its early-stop and
    # Top-K schedules produce on the staircase SPS table.  Here the early stop
    # lands just below the first cliff (B = 1024, b = 511); the Top-K budget,
    # the one a round kept from two rounds earlier, is taken as 3 R = 1536, a
    # budget past that cliff.
    wl = synth.WORKLOADS["r512_g16_v32768_staircase"]
    temperature, rnd = wl.temperatures[0], 0
    dr, inp = device_round(wl)
    W1, W2, w = weights(wl)
    every = np.arange(wl.R)
    drafted = oracle_draft(inp.U, W1, W2, inp.anchors, temperature, wl.seed, rnd, every)
    _, a = oracle_confidence(inp.h, W1, w, inp.anchors, drafted[0])
    sps = synth.sps_table(wl)
    early = oracle.schedule(a, sps, MODE_EARLY_STOP)
    topk = oracle.schedule(a, sps, MODE_TOP_K, 3 * wl.R)
    tokens, pd, lz, T, _ = verify_inputs(wl, inp, rnd, every, temperature, drafted=drafted)
    dr.T.copy_(torch.from_numpy(T))
    dr.tokens.copy_(torch.from_numpy(tokens))
    dr.pd.copy_(torch.from_numpy(pd))
    dr.logZ.copy_(torch.from_numpy(lz))
    seen = []
    for sched in (early, topk):
        lens = sched["lens"].astype(np.int32)
        assert 0 < lens.sum() < wl.R * wl.gamma and lens.min() < lens.max()  # ragged
        seen.append(tuple(lens))
        dr.lens.copy_(torch.from_numpy(lens))
        dr.verify(temperature, wl.seed, rnd)
        na, nx = host(dr.n_accept), host(dr.next_token)
        assert np.all(na >= 0) and np.all(na <= lens)
        ex = check_verify(wl, inp, T, tokens, lens, na, nx, temperature, rnd, every)
        assert ex <= wl.R // 8  # each exemption checked within tolerance
        assert dr.status() == 0
    assert seen[0] != seen[1]


def _run_c_star(wl, temperature, compare, lens=None, rnd=0):
    """Verify twice, without and with the analytic acceptance c*; the two
    calls must agree on every emitted token, and c* must match the oracle."""
    import oracle
    from gpu_helpers import PROB_TOL, weights
    dr, inp = device_round(wl)
    tokens, pd, lz, T, lens = verify_inputs(wl, inp, rnd, compare, temperature, lens)
    dr.T.copy_(torch.from_numpy(T))
    dr.tokens.copy_(torch.from_numpy(tokens))
    dr.pd.copy_(torch.from_numpy(pd))
    dr.logZ.copy_(torch.from_numpy(lz))
    dr.lens.copy_(torch.from_numpy(lens))
    dr.verify(temperature, wl.seed, rnd)
    na0, nx0 = host(dr.n_accept), host(dr.next_token)
    dr.c_star.fill_(-5.0)
    dr.verify(temperature, wl.seed, rnd, c_star=True)
    na, nx, cs = host(dr.n_accept), host(dr.next_token), host(dr.c_star)
    assert np.array_equal(na, na0) and np.array_equal(nx, nx0)
    assert dr.status() == 0
    # rows past lens[r] were not read: NaN there, a value everywhere else
    j = np.arange(wl.gamma)[None, :]
    assert np.array_equal(np.isnan(cs), j > lens[:, None])
    W1, W2, _ = weights(wl)
    cmp_ = np.asarray(compare)
    cs_o = oracle.c_star(T[cmp_], inp.U[cmp_], W1, W2, inp.anchors[cmp_], tokens[cmp_], lens[cmp_], temperature)
    got = cs[cmp_]
    assert np.array_equal(np.isnan(got), np.isnan(cs_o))
    m = ~np.isnan(cs_o)
    if temperature == 0.0:
        assert np.array_equal(got[m], cs_o[m])
    else:
        assert np.max(np.abs(got[m] - cs_o[m])) <= PROB_TOL
    ex = check_verify(wl, inp, T, tokens, lens, na, nx, temperature, rnd, compare)
    return cs, ex


@pytest.mark.parametrize("temperature", [1.0, 0.7, 0.0])
def test_c_star_tiny(temperature):
    _, ex = _run_c_star(TINY, temperature, range(TINY.R))
    assert ex <= 1


@pytest.mark.parametrize("temperature", [1.0, 0.0])
def test_c_star_ragged_lengths(temperature):
    wl = synth.scaled(TINY, R=9, gamma=5, V=1000, d=16, name="ragged_verify")
    lens = np.array([0, 1, 2, 3, 4, 5, 5, 0, 2], np.int32)
    _, ex = _run_c_star(wl, temperature, range(wl.R), lens=lens)
    assert ex <= 1


def test_c_star_many_mtiles():
    # 140 requests x up to 4 verify rows: residual rows over five M-tiles
    wl = synth.scaled(TINY, R=140, gamma=3, V=2048, rank=128, d=16, name="verify_r140")
    _, ex = _run_c_star(wl, 1.0, range(0, 140, 7))
    assert ex <= 1


def test_c_star_full_size():
    wl = synth.WORKLOADS["r128_g16_v151936"]
    rows = sample_requests(wl.R)
    _, ex = _run_c_star(wl, 1.0, rows)
    assert ex <= max(1, len(rows) // 4)
