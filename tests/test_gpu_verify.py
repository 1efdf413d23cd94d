"""GPU parity of dspark_verify against the oracle.  Draft outputs fed to
verify come from the oracle (compared requests) or stand-ins (the rest)."""
import numpy as np
import pytest
import torch

from gpu_helpers import check_verify, device_round, host, sample_requests, verify_inputs
from semi_autoregressive_speculative_gb300 import synth

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


def test_verify_many_rows_two_mtiles():
    wl = synth.scaled(TINY, R=140, gamma=3, V=2048, rank=128, d=16, name="verify_r140")
    na, nx, ex = _run(wl, 1.0, range(0, 140, 7))
    assert ex <= 1


@pytest.mark.parametrize("name", ["r32_g7_v151936", "r256_g16_v129280_d7168"])
def test_verify_full_size_sampled(name):
    wl = synth.WORKLOADS[name]
    for temperature in wl.temperatures:
        na, nx, ex = _run(wl, temperature, sample_requests(wl.R))
        assert ex <= 1
