"""Pins of the oracle's Markov-head draft ("DSpark" page §2.2-2.3).

Each test checks the oracle against something other than itself: a library
dense product, scipy's softmax plus numpy's inverse-CDF search when the
Markov head is zeroed (the draft then reduces to independent sampling),
a chi-square test of Philox draws against the exact distribution, and
numpy's first-occurrence argmax for greedy decoding.
"""
import numpy as np
import pytest
from scipy import special, stats

from semi_autoregressive_speculative_gb300 import synth


def _factors(rng, V, rank, std):
    W1 = synth.to_bf16_bits(rng.standard_normal((V, rank)).astype(np.float32) * std)
    W2 = synth.to_bf16_bits(rng.standard_normal((rank, V)).astype(np.float32) * std)
    return W1, W2


def _dense_bias(W1, W2):
    return synth.bf16_bits_to_f32(W1).astype(np.float64) @ synth.bf16_bits_to_f32(W2).astype(np.float64)


def test_bias_is_dense_product_row(orc):
    rng = np.random.default_rng(0)
    V, rank = 37, 16  # V != rank: a transposed operand cannot pass
    W1, W2 = _factors(rng, V, rank, 0.5)
    B = _dense_bias(W1, W2)
    for prev in (0, 5, 36):
        np.testing.assert_allclose(orc.markov_bias(W1, W2, prev), B[prev], rtol=0, atol=1e-12)


def test_probabilities_sum_to_one(orc):
    rng = np.random.default_rng(1)
    V, rank = 500, 32
    W1, W2 = _factors(rng, V, rank, 0.3)
    U = (rng.standard_normal(V) * 3).astype(np.float32)
    for T in (1.0, 0.7, 2.0):
        p, logZ = orc.draft_probs(U, W1, W2, 7, T)
        assert abs(p.sum() - 1.0) < 1e-12
        assert np.all(p > 0)


@pytest.mark.parametrize("zeroed", ["W1", "W2"])
@pytest.mark.parametrize("T", [1.0, 0.5])
def test_zero_markov_head_is_independent_sampling(orc, zeroed, T):
    rng = np.random.default_rng(2)
    V, rank, gamma = 50, 16, 5
    W1, W2 = _factors(rng, V, rank, 0.5)
    if zeroed == "W1":
        W1[:] = 0
    else:
        W2[:] = 0
    reqs = [4, 9, 11]
    U = (rng.standard_normal((3, gamma, V)) * 2).astype(np.float32)
    anchors = rng.integers(0, V, 3).astype(np.int32)
    tokens, pd, logZ = orc.draft(U, W1, W2, anchors, T, seed=3, rnd=2, request_ids=reqs)
    for i, r in enumerate(reqs):
        for j in range(gamma):
            z = U[i, j].astype(np.float64) / T
            p = special.softmax(z)
            u = orc.uniform(3, 2, r, j, 0)
            x = int(np.searchsorted(np.cumsum(p), u, side="right"))
            assert tokens[i, j] == x
            assert abs(pd[i, j] - p[x]) < 1e-6
            assert abs(logZ[i, j] - special.logsumexp(z)) < 1e-5


def test_each_position_conditions_on_previous_token(orc):
    # strong Markov head: the draft at position j follows softmax(U_j + B[x_{j-1}]),
    # x_{-1} = anchor; B from a library dense product
    rng = np.random.default_rng(3)
    V, rank, gamma = 40, 40, 6
    W1, W2 = _factors(rng, V, rank, 0.6)
    B = _dense_bias(W1, W2)
    U = rng.standard_normal((2, gamma, V)).astype(np.float32)
    anchors = np.array([3, 17], np.int32)
    tokens, pd, _ = orc.draft(U, W1, W2, anchors, 1.0, seed=8, rnd=0)
    differs = 0
    for i in range(2):
        prev = anchors[i]
        for j in range(gamma):
            p = special.softmax(U[i, j].astype(np.float64) + B[prev])
            u = orc.uniform(8, 0, i, j, 0)
            x = int(np.searchsorted(np.cumsum(p), u, side="right"))
            assert tokens[i, j] == x
            p0 = special.softmax(U[i, j].astype(np.float64))
            differs += int(np.searchsorted(np.cumsum(p0), u, side="right") != x)
            prev = x
    assert differs > 0  # the head actually changed some draws


def test_sampling_frequencies_chi_square(orc):
    rng = np.random.default_rng(4)
    V, rank, n = 8, 16, 100000
    W1, W2 = _factors(rng, V, rank, 0.5)
    U = rng.standard_normal(V).astype(np.float32)
    anchor = 3
    p = special.softmax(U.astype(np.float64) + _dense_bias(W1, W2)[anchor])
    Ub = np.broadcast_to(U, (n, 1, V)).copy()
    tokens, _, _ = orc.draft(Ub, W1, W2, np.full(n, anchor, np.int32), 1.0, seed=11, rnd=0)
    counts = np.bincount(tokens[:, 0], minlength=V)
    assert stats.chisquare(counts, p * n).pvalue > 1e-4


def test_greedy_lowest_index_on_ties(orc):
    V, rank = 16, 8
    W1 = np.zeros((V, rank), np.uint16)
    W2 = np.zeros((rank, V), np.uint16)
    U = np.zeros((1, 2, V), np.float32)
    U[0, 0, [5, 9]] = 3.0
    U[0, 1, [12, 2, 7]] = 1.5
    tokens, pd, logZ = orc.draft(U, W1, W2, [0], 0.0, seed=0, rnd=0)
    assert tokens.tolist() == [[5, 2]]
    assert pd.tolist() == [[1.0, 1.0]]


def test_greedy_is_first_argmax_of_fp32_logits(orc):
    rng = np.random.default_rng(5)
    V, rank, gamma = 300, 24, 5
    W1, W2 = _factors(rng, V, rank, 0.7)
    B = _dense_bias(W1, W2)
    U = rng.standard_normal((1, gamma, V)).astype(np.float32)
    tokens, _, _ = orc.draft(U, W1, W2, [11], 0.0, seed=0, rnd=0)
    prev = 11
    for j in range(gamma):
        z = (U[0, j].astype(np.float64) + B[prev]).astype(np.float32)
        assert tokens[0, j] == int(np.argmax(z))
        prev = tokens[0, j]
