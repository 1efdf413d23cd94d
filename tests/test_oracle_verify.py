"""Pins of the oracle's rejection-sampling verifier (standard speculative
verification, "DSpark" page introduction and §3.1 eq. c_k*).

* exact enumeration on a tiny vocabulary: with the accept and residual
  uniforms swept over fine grids, the first emitted token follows the target
  distribution;
* Monte Carlo over Philox rounds: the acceptance rate equals the overlap
  1 - 0.5 ||p_d - p_t||_1, and with two draft positions the second emitted
  token, given the first, follows the target's conditional row;
* greedy decoding is the exact special case (accept iff the draft token is
  the target argmax; the next token is the argmax of the first rejected row).
"""
import numpy as np
from scipy import special, stats

from semi_autoregressive_speculative_gb300 import synth


def _tiny(rng, V, rank, gamma, std=0.8):
    W1 = synth.to_bf16_bits(rng.standard_normal((V, rank)).astype(np.float32) * std)
    W2 = synth.to_bf16_bits(rng.standard_normal((rank, V)).astype(np.float32) * std)
    U = rng.standard_normal((gamma, V)).astype(np.float32)
    return W1, W2, U


def test_overlap_is_sum_of_minimum(orc):
    rng = np.random.default_rng(0)
    for _ in range(10):
        p = special.softmax(rng.standard_normal(9))
        q = special.softmax(rng.standard_normal(9))
        assert abs(orc.overlap(p, q) - np.minimum(p, q).sum()) < 1e-12


def test_first_token_follows_target_exact_enumeration(orc):
    rng = np.random.default_rng(1)
    V, rank, N = 3, 4, 240
    W1, W2, U = _tiny(rng, V, rank, 1)
    anchor = 2
    T = rng.standard_normal((2, V)).astype(np.float32) * 1.5
    pd, _ = orc.draft_probs(U[0], W1, W2, anchor, 1.0)
    pt, _ = orc.target_probs(T[0], 1.0)
    grid = (np.arange(N) + 0.5) / N
    dist = np.zeros(V)
    for x in range(V):
        counts = np.zeros(V)
        for ua in grid:
            for ur in grid:
                na, nxt = orc.verify_request_u(T, U, W1, W2, anchor, [x], 1, 1.0, [ua], [ur, ur])
                first = x if na == 1 else nxt
                counts[first] += 1
        dist += pd[x] * counts / N**2
    np.testing.assert_allclose(dist, pt, atol=3.0 / N)


def test_acceptance_rate_is_overlap(orc):
    rng = np.random.default_rng(2)
    V, rank, n = 8, 8, 40000
    W1, W2, U = _tiny(rng, V, rank, 1, 0.4)
    T = (U + rng.standard_normal((1, V)).astype(np.float32))
    T = np.concatenate([T, rng.standard_normal((1, V)).astype(np.float32)])[None]
    pd, _ = orc.draft_probs(U[0], W1, W2, 0, 1.0)
    pt, _ = orc.target_probs(T[0, 0], 1.0)
    alpha = orc.overlap(pd, pt)
    acc = np.empty(n)
    first = np.empty(n, np.int64)
    bonus = []
    for rnd in range(n):
        tok, _, _ = orc.draft(U[None], W1, W2, [0], 1.0, seed=7, rnd=rnd)
        na, nxt = orc.verify(T, U[None], W1, W2, [0], tok, [1], 1.0, seed=7, rnd=rnd)
        acc[rnd] = na[0]
        first[rnd] = tok[0, 0] if na[0] == 1 else nxt[0]
        if na[0] == 1:
            bonus.append(nxt[0])
    assert abs(acc.mean() - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / n)
    counts = np.bincount(first, minlength=V)
    assert stats.chisquare(counts, pt * n).pvalue > 1e-4
    # after a full accept the bonus token follows the target's next row
    pb, _ = orc.target_probs(T[0, 1], 1.0)
    nb = len(bonus)
    assert stats.chisquare(np.bincount(bonus, minlength=V), pb * nb).pvalue > 1e-4


def test_second_token_follows_target_conditional(orc):
    # gamma = 2; the target's row for position 2 depends on the first draft
    # token (L[x1]); given that the first token was accepted as v1, the second
    # emitted token must follow softmax(L[v1]).
    rng = np.random.default_rng(3)
    V, rank, n = 3, 4, 60000
    W1, W2, U = _tiny(rng, V, rank, 2, 0.9)
    T0 = rng.standard_normal(V).astype(np.float32)
    L = rng.standard_normal((V, V)).astype(np.float32) * 1.5
    Bon = rng.standard_normal((V, V)).astype(np.float32)
    anchor = 1
    pairs = {v: [] for v in range(V)}
    firsts = []
    for rnd in range(n):
        tok, _, _ = orc.draft(U[None], W1, W2, [anchor], 1.0, seed=9, rnd=rnd)
        x1, x2 = int(tok[0, 0]), int(tok[0, 1])
        T = np.stack([T0, L[x1], Bon[x2]])[None]
        na, nxt = orc.verify(T, U[None], W1, W2, [anchor], tok, [2], 1.0, seed=9, rnd=rnd)
        na = int(na[0])
        emitted = [x1, x2][:na] + [int(nxt[0])]
        firsts.append(emitted[0])
        if len(emitted) >= 2:
            pairs[emitted[0]].append(emitted[1])
    pt0 = special.softmax(T0.astype(np.float64))
    assert stats.chisquare(np.bincount(firsts, minlength=V), pt0 * n).pvalue > 1e-4
    for v1 in range(V):
        seconds = np.array(pairs[v1])
        if len(seconds) < 500:
            continue
        p2 = special.softmax(L[v1].astype(np.float64))
        assert stats.chisquare(np.bincount(seconds, minlength=V), p2 * len(seconds)).pvalue > 1e-4


def test_certain_accept_and_certain_reject_rows(orc):
    # position 0: the target puts all mass where the draft does (ratio >= 1,
    # always accepted); position 1: the target gives the draft token no mass
    # (always rejected); the residual then follows the target row 1.
    rng = np.random.default_rng(4)
    V, rank = 5, 4
    W1 = np.zeros((V, rank), np.uint16)
    W2 = np.zeros((rank, V), np.uint16)
    U = np.zeros((3, V), np.float32)
    U[0, 2] = 30.0
    tokens = np.array([2, 4, 0], np.int32)
    T = rng.standard_normal((4, V)).astype(np.float32)
    T[0, 2] = 60.0
    T[1, 4] = -200.0
    n = 3000
    nxt_all = np.empty(n, np.int64)
    for rnd in range(n):
        na, nxt = orc.verify(T[None], U[None], W1, W2, [0], tokens[None], [3], 1.0, seed=1, rnd=rnd)
        assert na[0] == 1
        nxt_all[rnd] = nxt[0]
    # residual at position 1: max(0, p_t - p_d) renormalised, p_d uniform here
    q = np.maximum(0.0, special.softmax(T[1].astype(np.float64)) - 1.0 / V)
    q /= q.sum()
    counts = np.bincount(nxt_all, minlength=V)
    assert np.all(counts[q == 0] == 0)
    keep = q > 0
    assert stats.chisquare(counts[keep], q[keep] * n).pvalue > 1e-4


def test_greedy_special_case(orc):
    V, rank = 6, 4
    W1 = np.zeros((V, rank), np.uint16)
    W2 = np.zeros((rank, V), np.uint16)
    U = np.zeros((3, V), np.float32)
    T = np.zeros((4, V), np.float32)
    T[0, 3] = T[0, 1] = 2.0      # tie: argmax is 1
    T[1, 5] = 1.0
    T[2, 0] = 1.0
    T[3, 2] = 1.0
    cases = [([1, 5, 0], 3, 3, 2), ([1, 5, 4], 3, 2, 0), ([3, 5, 0], 3, 0, 1), ([1, 5, 0], 2, 2, 0),
             ([1, 5, 0], 0, 0, 1)]
    for toks, length, n_acc, nxt in cases:
        na, nx = orc.verify(T[None], U[None], W1, W2, [0], np.array([toks], np.int32), [length],
                            0.0, seed=0, rnd=0)
        assert (na[0], nx[0]) == (n_acc, nxt)


def test_c_star_is_the_acceptance_probability(orc):
    # c*_j ("DSpark" §3.1, eq. c_k*) is the chance that verification accepts
    # position j given an accepted prefix: E_{x ~ p_d}[min(1, p_t(x) / p_d(x))].
    # Measured here on the verifier itself, sweeping its accept uniform over a
    # fine grid for every candidate x at position j; the prefix is accepted by
    # giving it u = 0.
    rng = np.random.default_rng(11)
    V, rank, gamma, N = 5, 4, 3, 400
    W1, W2, U = _tiny(rng, V, rank, gamma)
    T = (rng.standard_normal((gamma + 1, V)) * 1.3).astype(np.float32)
    anchor, temp = 1, 0.8
    prefix = np.array([3, 0, 0], np.int32)
    cs = orc.c_star(T[None], U[None], W1, W2, [anchor], prefix[None], [gamma], temp)[0]
    grid = (np.arange(N) + 0.5) / N
    for j in range(gamma):
        prev = anchor if j == 0 else int(prefix[j - 1])
        pd, _ = orc.draft_probs(U[j], W1, W2, prev, temp)
        expect = 0.0
        for x in range(V):
            toks = prefix.copy()
            toks[j] = x
            acc = 0
            for ua in grid:
                u_acc = np.zeros(gamma)
                u_acc[j] = ua
                na, _ = orc.verify_request_u(T, U, W1, W2, anchor, toks, j + 1, temp, u_acc, np.full(gamma + 1, 0.5))
                acc += na == j + 1
            expect += pd[x] * acc / N
        assert abs(cs[j] - expect) <= 1.0 / N


def test_c_star_rows_identity_and_greedy(orc):
    rng = np.random.default_rng(12)
    V, rank, gamma = 7, 4, 4
    W1, W2, U = _tiny(rng, V, rank, gamma)
    anchor = 2
    toks = np.array([[1, 6, 0, 3]], np.int32)
    # target rows equal to the draft logits: the distributions coincide, c* = 1
    T = np.empty((gamma + 1, V), np.float32)
    for j in range(gamma):
        prev = anchor if j == 0 else int(toks[0, j - 1])
        T[j] = orc.draft_logits_f32(U[j], W1, W2, prev)
    T[gamma] = 0.0
    for length in range(gamma + 1):
        cs = orc.c_star(T[None], U[None], W1, W2, [anchor], toks, [length], 1.3)[0]
        last = min(length, gamma - 1)
        np.testing.assert_allclose(cs[: last + 1], 1.0, atol=1e-6)
        assert np.all(np.isnan(cs[last + 1:]))  # positions past the verified rows
    # greedy: 1 where the drafted token is the target's first argmax, else 0
    Tg = rng.standard_normal((gamma + 1, V)).astype(np.float32)
    Tg[1, 6] = Tg[1].max() + 1.0
    Tg[2, 4] = Tg[2, 0] = Tg[2].max() + 1.0  # tie: the argmax is 0
    cs = orc.c_star(Tg[None], U[None], W1, W2, [anchor], toks, [3], 0.0)[0]
    expect = [float(toks[0, j] == int(np.argmax(Tg[j]))) for j in range(4)]
    np.testing.assert_array_equal(cs, expect)
    assert cs[1] == 1.0 and cs[2] == 1.0
