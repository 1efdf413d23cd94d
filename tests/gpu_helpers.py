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
import os
from concurrent.futures import ThreadPoolExecutor

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


# ------------------------------------------------------------------ the oracle on many requests
# The oracle is single-threaded C behind ctypes, which releases the GIL during
# each call, and it keeps no global state: independent requests run on a
# thread pool, one oracle call per request, with the oracle's own code and
# arithmetic unchanged.
_POOL = None


def pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        oracle.lib()  # build and load once, before any worker thread calls it
        _POOL = ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))
    return _POOL


def par_map(fn, items):
    return list(pool().map(fn, list(items)))


def oracle_draft(U, W1, W2, anchors, temperature, seed, rnd, request_ids):
    """oracle.draft over rows of U (row i is request request_ids[i])."""
    req = np.asarray(request_ids)
    anchors = np.asarray(anchors, np.int32)

    def one(i):
        return oracle.draft(U[i:i + 1], W1, W2, anchors[i:i + 1], temperature, seed, rnd, request_ids=req[i:i + 1])
    outs = par_map(one, range(len(req)))
    return tuple(np.concatenate([o[k] for o in outs]) for k in range(3))


def oracle_verify(T, U, W1, W2, anchors, tokens, lens, temperature, seed, rnd, request_ids):
    req = np.asarray(request_ids)

    def one(i):
        return oracle.verify(T[i:i + 1], U[i:i + 1], W1, W2, np.asarray(anchors[i:i + 1], np.int32),
                             tokens[i:i + 1], lens[i:i + 1], temperature, seed, rnd, request_ids=req[i:i + 1])
    outs = par_map(one, range(len(req)))
    return np.concatenate([o[0] for o in outs]), np.concatenate([o[1] for o in outs])


def oracle_confidence(h, W1, w, anchors, tokens):
    def one(i):
        return oracle.confidence(h[i:i + 1], W1, w, np.asarray(anchors[i:i + 1], np.int32), tokens[i:i + 1])
    outs = par_map(one, range(h.shape[0]))
    return np.concatenate([o[0] for o in outs]), np.concatenate([o[1] for o in outs])


def prefix_bias(W1, W2, anchor, tokens_r):
    """Oracle Markov bias [gamma, V] of each position of one request, from its
    drafted prefix (the anchor, then tokens_r[:-1])."""
    prevs = [int(anchor)] + [int(x) for x in tokens_r[:-1]]
    return np.stack(par_map(lambda pv: oracle.markov_bias(W1, W2, pv), prevs))


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
def _inverse_cdf_legit(p, x, u, tol=CDF_TOL):
    """x is the inverse-CDF draw of some u' within tol of u."""
    cdf = np.cumsum(p)
    lo = cdf[x - 1] if x > 0 else 0.0
    return lo - tol <= u < cdf[x] + tol


def check_draft(wl, inp, tok_g, pd_g, lz_g, temperature, rnd, requests, counts=None, cdf_tol=CDF_TOL,
                logz_tol=LOGZ_TOL, tie_tol=1e-4):
    """Compare GPU draft outputs of `requests` with the oracle's.  Returns the
    number of legitimate divergences and of near-tie greedy rows; `counts`
    (a dict), when given, receives the number of draws compared.

    At full vocabulary the draft distributions are flat (151936 tokens, most
    with probability 1e-6 to 1e-5), so a token's CDF interval is often
    narrower than the fp32 error of the kernel's cumulative sums, and a draw
    within 1e-5 of a boundary may legitimately pick a neighbour.  The
    tolerances (CDF, log Z, greedy near-tie gap) default to the draft's own;
    the fused LM-head draft passes wider ones derived from its longer fp32
    sums."""
    W1, W2, _ = weights(wl)
    req = np.asarray(requests)
    tok_o, pd_o, lz_o = oracle_draft(inp.U[req], W1, W2, inp.anchors[req], temperature, wl.seed, rnd, req)
    diverged = near_ties = compared = 0
    for i, r in enumerate(req):
        prev = int(inp.anchors[r])
        for j in range(wl.gamma):
            compared += 1
            xg, xo = int(tok_g[r, j]), int(tok_o[i, j])
            if temperature == 0.0:
                if xg != xo:
                    z = oracle.draft_logits_f32(inp.U[r, j], W1, W2, prev)
                    top2 = np.sort(z)[-2:]
                    assert top2[1] - top2[0] < tie_tol, f"greedy token differs at r={r} j={j}: {xg} vs {xo}"
                    near_ties += 1
                    break
                assert pd_g[r, j] == 1.0
                assert abs(lz_g[r, j] - lz_o[i, j]) <= logz_tol * max(1.0, abs(lz_o[i, j]))
            else:
                if xg != xo:
                    p, _ = oracle.draft_probs(inp.U[r, j], W1, W2, prev, temperature)
                    u = oracle.uniform(wl.seed, rnd, int(r), j, 0)
                    assert _inverse_cdf_legit(p, xg, u, cdf_tol), \
                        f"sampled token differs at r={r} j={j}: gpu {xg} oracle {xo}, u={u}"
                    diverged += 1
                    break
                assert abs(pd_g[r, j] - pd_o[i, j]) <= PROB_TOL, (r, j, pd_g[r, j], pd_o[i, j])
                assert abs(lz_g[r, j] - lz_o[i, j]) <= logz_tol * max(1.0, abs(lz_o[i, j])), \
                    (r, j, lz_g[r, j], lz_o[i, j])
            prev = xo
    if counts is not None:
        counts["compared"] = compared
    return diverged, near_ties


def check_draft_forced(wl, U_rows, anchors, tok_g, pd_g, lz_g, temperature, rnd, requests, cdf_tol=CDF_TOL,
                       logz_tol=LOGZ_TOL, tie_tol=1e-4, prob_tol=PROB_TOL):
    """Every position of every request in `requests` against the oracle's
    distribution conditioned on the kernel's own previous token (teacher
    forcing), so that a legitimate divergence early in a row does not end
    the comparison of that row.  U_rows[r] is request r's U [gamma, V].  Each
    drawn token must be the oracle's inverse-CDF draw of the same Philox u, or
    one whose CDF interval lies within cdf_tol of u; greedy: the oracle's
    argmax, or within tie_tol of it.  p_d and log Z are compared at every
    position.  Returns the number of draws that differ from the oracle's."""
    W1, W2, _ = weights(wl)

    def one(r):
        differ = 0
        prev = int(anchors[r])
        for j in range(wl.gamma):
            xg = int(tok_g[r, j])
            if temperature == 0.0:
                z = oracle.draft_logits_f32(U_rows[r][j], W1, W2, prev)
                xo = int(np.argmax(z))
                if xg != xo:
                    assert z[xo] - z[xg] < tie_tol, f"greedy token at r={r} j={j}: {xg} vs {xo}"
                    differ += 1
                assert pd_g[r, j] == 1.0
                assert abs(lz_g[r, j] - float(z[xg])) <= logz_tol * max(1.0, abs(float(z[xg]))), (r, j)
            else:
                p, logZ = oracle.draft_probs(U_rows[r][j], W1, W2, prev, temperature)
                u = oracle.uniform(wl.seed, rnd, int(r), j, 0)
                xo = oracle.inverse_cdf(p, u)
                if xg != xo:
                    assert _inverse_cdf_legit(p, xg, u, cdf_tol), f"sampled token at r={r} j={j}: {xg} vs {xo}, u={u}"
                    differ += 1
                assert abs(pd_g[r, j] - p[xg]) <= prob_tol, (r, j, pd_g[r, j], p[xg])
                assert abs(lz_g[r, j] - logZ) <= logz_tol * max(1.0, abs(logZ)), (r, j, lz_g[r, j], logZ)
            prev = xg
        return differ
    return sum(par_map(one, [int(r) for r in requests]))


# ------------------------------------------------------------------ verify inputs
def verify_inputs(wl, inp, rnd, compare, temperature, lens=None, drafted=None):
    """Draft outputs fed to verify: the oracle's draft for the `compare`
    requests (`drafted`, when the caller already has it), stand-in values for
    the rest; target logits T = U + Markov bias of the fed prefix + noise
    (bias from the oracle for compared requests; the stand-in rows skip it)."""
    W1, W2, _ = weights(wl)
    R, g, V = wl.R, wl.gamma, wl.V
    tokens = np.empty((R, g), np.int32)
    pd = np.empty((R, g), np.float32)
    lz = np.empty((R, g), np.float32)
    for r in range(R):
        tokens[r], pd[r], lz[r] = synth.fake_draft(wl, rnd, r)
    cmp_ = np.asarray(compare)
    if drafted is None:
        drafted = oracle_draft(inp.U[cmp_], W1, W2, inp.anchors[cmp_], temperature, wl.seed, rnd, cmp_)
    t_o, p_o, z_o = drafted
    tokens[cmp_], pd[cmp_], lz[cmp_] = t_o, p_o, z_o
    T = np.empty((R, g + 1, V), np.float32)
    cset = set(int(c) for c in cmp_)
    for r in range(R):
        noise = synth.target_noise(wl, rnd, r)
        if r in cset:
            bias = prefix_bias(W1, W2, inp.anchors[r], tokens[r])
        else:
            bias = np.zeros((g, V))
        T[r] = synth.compose_target(inp.U[r], bias, noise, synth.bonus_base(wl, rnd, r))
    if lens is None:
        lens = np.full(R, g, np.int32)
    return tokens, pd, lz, T, np.asarray(lens, np.int32)


def check_verify(wl, inp, T, tokens, lens, na_g, nx_g, temperature, rnd, compare):
    W1, W2, _ = weights(wl)
    cmp_ = np.asarray(compare)
    na_o, nx_o = oracle_verify(T[cmp_], inp.U[cmp_], W1, W2, inp.anchors[cmp_], tokens[cmp_], lens[cmp_],
                               temperature, wl.seed, rnd, cmp_)
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


def sample_requests(R):
    """Requests compared at full size: the first, a middle and the last row of
    every 32-row lane quarter of every 128-row M-tile (each quarter is read from
    tensor memory by its own epilogue warps, and every M-tile has its own
    ready counter, chunk entries and A-operand staging), plus the last
    request."""
    rows = set()
    for m0 in range(0, R, 128):
        for q0 in range(m0, min(R, m0 + 128), 32):
            q1 = min(R, q0 + 32)
            rows.update((q0, (q0 + q1) // 2, q1 - 1))
    rows.add(R - 1)
    return sorted(rows)


requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
