"""Pins of the oracle's confidence head and survival products
("DSpark" page §3.1 eq. c_k, §1.1 eq. a_j and eq. tau)."""
import numpy as np

from semi_autoregressive_speculative_gb300 import synth


def test_closed_form_tiny_head(orc):
    # d = 4, r = 2, V = 3; w = [w_h (4) ; w_e (2)]
    h = synth.to_bf16_bits(np.array([[[1.0, 0.0, 0.0, 0.0], [0.0, 2.0, 0.0, 0.0]]], np.float32))
    w = np.array([0.5, 0.25, 0.0, 0.0, 2.0, -1.0], np.float32)
    W1 = synth.to_bf16_bits(np.array([[0.25, 0.0], [0.0, 0.5], [1.0, 1.0]], np.float32))
    anchor, tokens = 1, np.array([[2, 0]], np.int32)
    c, a = orc.confidence(h, W1, w, [anchor], tokens)
    # position 0 reads the anchor's row: s = 0.5*1 + (2*0 - 1*0.5) = 0      -> sigma(0) = 1/2
    # position 1 reads token 0's row:     s = 0.25*2 + (2*1 - 1*1) = 1.5   -> sigma(1.5)
    sig15 = 1.0 / (1.0 + np.exp(-1.5))
    assert c[0, 0] == np.float32(0.5)
    assert abs(c[0, 1] - sig15) < 1e-7
    assert a[0, 0] == c[0, 0]
    assert a[0, 1] == np.float32(c[0, 0] * c[0, 1])


def test_matches_library_logistic(orc):
    from scipy import special
    rng = np.random.default_rng(0)
    V, rank, d, gamma, n = 50, 16, 40, 6, 4
    W1 = synth.to_bf16_bits(rng.standard_normal((V, rank)).astype(np.float32) * 0.3)
    h = synth.to_bf16_bits(rng.standard_normal((n, gamma, d)).astype(np.float32))
    w = (rng.standard_normal(d + rank) * 0.2).astype(np.float32)
    anchors = rng.integers(0, V, n).astype(np.int32)
    tokens = rng.integers(0, V, (n, gamma)).astype(np.int32)
    c, a = orc.confidence(h, W1, w, anchors, tokens)
    hf = synth.bf16_bits_to_f32(h).astype(np.float64)
    Ef = synth.bf16_bits_to_f32(W1).astype(np.float64)
    for i in range(n):
        prev = np.concatenate([[anchors[i]], tokens[i, :-1]])
        s = hf[i] @ w[:d].astype(np.float64) + Ef[prev] @ w[d:].astype(np.float64)
        np.testing.assert_allclose(c[i], special.expit(s).astype(np.float32), rtol=0, atol=1e-7)
        np.testing.assert_array_equal(a[i], np.cumprod(c[i], dtype=np.float32))
        assert np.all(np.diff(a[i]) <= 0)


def test_survival_is_running_fp32_product(orc):
    rng = np.random.default_rng(1)
    c = rng.uniform(0, 1, (7, 13)).astype(np.float32)
    c[0, 3] = 1.0
    c[1, 5] = 0.0
    a = orc.survival(c)
    np.testing.assert_array_equal(a, np.cumprod(c, axis=1, dtype=np.float32))
    assert np.all(np.diff(a, axis=1) <= 0)


def test_tau_is_expected_emitted_tokens(orc):
    # When position j is accepted with probability c_j given all earlier ones
    # were, the expected tokens per round (accepted drafts + the one the
    # verifier adds) is tau = 1 + sum_j a_j ("DSpark" page §1.1).  Build draft
    # and target rows whose per-position acceptance is independent of the
    # prefix (zero Markov head), set c_j to the analytic overlap, and compare
    # tau with the verifier's empirical mean.
    rng = np.random.default_rng(2)
    V, rank, gamma, n = 6, 4, 3, 30000
    W1 = np.zeros((V, rank), np.uint16)
    W2 = np.zeros((rank, V), np.uint16)
    U = rng.standard_normal((1, gamma, V)).astype(np.float32)
    T = (U[0] + 0.8 * rng.standard_normal((gamma, V))).astype(np.float32)
    T = np.concatenate([T, rng.standard_normal((1, V)).astype(np.float32)])[None]
    c = np.array([orc.overlap(orc.draft_probs(U[0, j], W1, W2, 0, 1.0)[0],
                              orc.target_probs(T[0, j], 1.0)[0]) for j in range(gamma)], np.float32)
    tau = 1.0 + float(orc.survival(c).astype(np.float64).sum())
    emitted = np.empty(n)
    for rnd in range(n):
        tok, _, _ = orc.draft(U, W1, W2, [0], 1.0, seed=5, rnd=rnd)
        na, _ = orc.verify(T, U, W1, W2, [0], tok, [gamma], 1.0, seed=5, rnd=rnd)
        emitted[rnd] = na[0] + 1
    se = emitted.std() / np.sqrt(n)
    assert abs(emitted.mean() - tau) < 4 * se


def test_sts_temperatures_divide_the_logits(orc):
    # sequential temperature scaling ("DSpark" page §3.2): c_j = sigma(s_j / t_j)
    from scipy import special
    rng = np.random.default_rng(3)
    V, rank, d, gamma, n = 40, 16, 24, 5, 3
    W1 = synth.to_bf16_bits(rng.standard_normal((V, rank)).astype(np.float32) * 0.5)
    h = synth.to_bf16_bits(rng.standard_normal((n, gamma, d)).astype(np.float32))
    w = (rng.standard_normal(d + rank) * 0.3).astype(np.float32)
    anchors = rng.integers(0, V, n).astype(np.int32)
    tokens = rng.integers(0, V, (n, gamma)).astype(np.int32)
    t = np.array([1.0, 0.5, 2.0, 3.0, 0.25], np.float32)
    c1, _ = orc.confidence(h, W1, w, anchors, tokens)
    cu, au = orc.confidence(h, W1, w, anchors, tokens, sts_temperature=np.ones(gamma, np.float32))
    np.testing.assert_array_equal(cu, c1)  # unit temperatures change nothing
    ct, at = orc.confidence(h, W1, w, anchors, tokens, sts_temperature=t)
    logit = np.log(c1.astype(np.float64)) - np.log1p(-c1.astype(np.float64))
    np.testing.assert_allclose(ct, special.expit(logit / t.astype(np.float64)), atol=2e-7)
    np.testing.assert_array_equal(at, np.cumprod(ct, axis=1, dtype=np.float32))
    # t > 1 pulls a confidence towards 1/2, t < 1 away from it
    hot, cold = t > 1, t < 1
    assert np.all(np.abs(ct[:, hot] - 0.5) <= np.abs(c1[:, hot] - 0.5) + 1e-7)
    assert np.all(np.abs(ct[:, cold] - 0.5) >= np.abs(c1[:, cold] - 0.5) - 1e-7)
