"""Shared machinery of the GPU parity tests: seeded inputs of a workload, the
device round, and the comparison rules against the CPU oracle.

Tolerances (fixed by the project's statement of the hot path):
  * tokens, scheduler lengths and accept counts bit-exact when greedy, and
    scheduler outputs bit-exact when both sides get the same a;
  * probabilities and confidences within 1e-4 absolute;
  * a sampled token may differ only where |CDF - u| < 1e-5: the GPU's token
    must be the inverse-CDF draw of some u' with |u' - u| < 1e-5 under the
    oracle's distribution; an accept decision may differ only where
    |u - p_t/p_d| < 1e-5.  After such a divergence the request's later
    positions condition on different prefixes and are not compared.
No input of the oracle ever comes from the CUDA path.
"""
from __future__ import annotations

import functools

import numpy as np
import pytest
import torch

import oracle
from semi_autoregressive_speculative_gb300 import synth

PROB_TOL = 1e-4
CDF_TOL = 1e-5
LOGZ_TOL = 1e-4


@functools.lru_cache(maxsize=4)
def weights(wl: synth.Workload):
    return synth.weights(wl)


def round_inputs(wl, rnd=0):
    return synth.round_inputs(wl, rnd)


def device_round(wl, inp=None, rnd=0):
    from semi_autoregressive_speculative_gb300.round import DeviceRound
    W1, W2, w = weights(wl)
    inp = inp or round_inputs(wl, rnd)
    dr = DeviceRound(wl.R, wl.gamma, wl.V, wl.rank, wl.d)
    dr.set_weights(W1, W2, w)
    dr.set_round(inp.U, inp.h, inp.anchors, synth.sps_table(wl))
    dr.clear_status()
    return dr, inp


def host(t):
    torch.cuda.synchronize()
    return t.detach().cpu().numpy()


# ------------------------------------------------------------------ draft
def _inverse_cdf_legit(p, x, u):
    """x is the inverse-CDF draw of some u' within CDF_TOL of u."""
    cdf = np.cumsum(p)
    lo = cdf[x - 1] if x > 0 else 0.0
    return lo - CDF_TOL <= u < cdf[x] + CDF_TOL


def check_draft(wl, inp, tok_g, pd_g, lz_g, temperature, rnd, requests):
    """Compare GPU draft outputs of `requests` with the oracle's.  Returns the
    number of legitimate divergences and of near-tie greedy rows."""
    W1, W2, _ = weights(wl)
    req = np.asarray(requests)
    tok_o, pd_o, lz_o = oracle.draft(inp.U[req], W1, W2, inp.anchors[req], temperature, wl.seed, rnd,
                                     request_ids=req)
    diverged = near_ties = 0
    for i, r in enumerate(req):
        prev = int(inp.anchors[r])
        for j in range(wl.gamma):
            xg, xo = int(tok_g[r, j]), int(tok_o[i, j])
            if temperature == 0.0:
                if xg != xo:
                    z = oracle.draft_logits_f32(inp.U[r, j], W1, W2, prev)
                    top2 = np.sort(z)[-2:]
                    assert top2[1] - top2[0] < 1e-4, f"greedy token differs at r={r} j={j}: {xg} vs {xo}"
                    near_ties += 1
                    break
                assert pd_g[r, j] == 1.0
                assert abs(lz_g[r, j] - lz_o[i, j]) <= LOGZ_TOL * max(1.0, abs(lz_o[i, j]))
            else:
                if xg != xo:
                    p, _ = oracle.draft_probs(inp.U[r, j], W1, W2, prev, temperature)
                    u = oracle.uniform(wl.seed, rnd, int(r), j, 0)
                    assert _inverse_cdf_legit(p, xg, u), \
                        f"sampled token differs at r={r} j={j}: gpu {xg} oracle {xo}, u={u}"
                    diverged += 1
                    break
                assert abs(pd_g[r, j] - pd_o[i, j]) <= PROB_TOL, (r, j, pd_g[r, j], pd_o[i, j])
                assert abs(lz_g[r, j] - lz_o[i, j]) <= LOGZ_TOL * max(1.0, abs(lz_o[i, j])), \
                    (r, j, lz_g[r, j], lz_o[i, j])
            prev = xo
    return diverged, near_ties


# ------------------------------------------------------------------ verify inputs
def verify_inputs(wl, inp, rnd, compare, temperature, lens=None):
    """Draft outputs fed to verify: the oracle's draft for the `compare`
    requests, stand-in values for the rest; target logits T = U + Markov bias
    of the fed prefix + noise (bias from the oracle for compared requests;
    the stand-in rows skip it)."""
    W1, W2, _ = weights(wl)
    R, g, V = wl.R, wl.gamma, wl.V
    tokens = np.empty((R, g), np.int32)
    pd = np.empty((R, g), np.float32)
    lz = np.empty((R, g), np.float32)
    for r in range(R):
        tokens[r], pd[r], lz[r] = synth.fake_draft(wl, rnd, r)
    cmp_ = np.asarray(compare)
    t_o, p_o, z_o = oracle.draft(inp.U[cmp_], W1, W2, inp.anchors[cmp_], temperature, wl.seed, rnd,
                                 request_ids=cmp_)
    tokens[cmp_], pd[cmp_], lz[cmp_] = t_o, p_o, z_o
    T = np.empty((R, g + 1, V), np.float32)
    cset = set(int(c) for c in cmp_)
    for r in range(R):
        noise = synth.target_noise(wl, rnd, r)
        if r in cset:
            prevs = [int(inp.anchors[r])] + [int(x) for x in tokens[r, :-1]]
            bias = np.stack([oracle.markov_bias(W1, W2, pv) for pv in prevs])
        else:
            bias = np.zeros((g, V))
        T[r] = synth.compose_target(inp.U[r], bias, noise, synth.bonus_base(wl, rnd, r))
    if lens is None:
        lens = np.full(R, g, np.int32)
    return tokens, pd, lz, T, np.asarray(lens, np.int32)


def check_verify(wl, inp, T, tokens, lens, na_g, nx_g, temperature, rnd, compare):
    W1, W2, _ = weights(wl)
    cmp_ = np.asarray(compare)
    na_o, nx_o = oracle.verify(T[cmp_], inp.U[cmp_], W1, W2, inp.anchors[cmp_], tokens[cmp_], lens[cmp_],
                               temperature, wl.seed, rnd, request_ids=cmp_)
    exempt = 0
    for i, r in enumerate(cmp_):
        if temperature == 0.0:
            assert na_g[r] == na_o[i] and nx_g[r] == nx_o[i], (r, na_g[r], na_o[i], nx_g[r], nx_o[i])
            continue
        if na_g[r] != na_o[i]:
            j = min(na_g[r], na_o[i])
            prev = int(inp.anchors[r]) if j == 0 else int(tokens[r, j - 1])
            pt, _ = oracle.target_probs(T[r, j], temperature)
            pdist, _ = oracle.draft_probs(inp.U[r, j], W1, W2, prev, temperature)
            x = int(tokens[r, j])
            u = oracle.uniform(wl.seed, rnd, int(r), j, 1)
            assert abs(u - pt[x] / pdist[x]) < CDF_TOL, (r, j, u, pt[x] / pdist[x], na_g[r], na_o[i])
            exempt += 1
            continue
        n = int(na_o[i])
        if nx_g[r] != nx_o[i]:
            pt, _ = oracle.target_probs(T[r, n], temperature)
            if n < lens[r]:
                prev = int(inp.anchors[r]) if n == 0 else int(tokens[r, n - 1])
                pdist, _ = oracle.draft_probs(inp.U[r, n], W1, W2, prev, temperature)
                q = np.maximum(pt - pdist, 0.0)
                dist = q / q.sum() if q.sum() > 0 else pt
            else:
                dist = pt
            u = oracle.uniform(wl.seed, rnd, int(r), n, 2)
            assert _inverse_cdf_legit(dist, int(nx_g[r]), u), (r, n, nx_g[r], nx_o[i], u)
            exempt += 1
    return exempt


def sample_requests(R, k=3):
    if R <= k:
        return list(range(R))
    return sorted(set([0, R // 2, R - 1] + list(range(1, k - 2))))


requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
