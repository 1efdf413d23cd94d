"""The fused LM-head draft (dspark_markov_draft_lmhead) against the oracle.

The oracle forms U = h . W_lm (oracle.lm_head_logits: fp64 sums rounded once
to fp32) and drafts from it exactly as for a given U; the kernel instead sums
the d LM-head products and the rank bias products in one fp32 tensor-core
accumulation.  One fp32 sum over d + rank = 4352 products of logits of size
about 3 to 10 carries an error of about sqrt(d + rank) * 2^-24 times the
running sum, about 2e-5, so the comparison allows 5e-4 on log Z and on the
greedy top-two gap and 1e-4 on the CDF; p_d keeps its 1e-4.
"""
import types

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import PROB_TOL, check_draft, host, sample_requests
from semi_autoregressive_speculative_gb300 import synth

LM_CDF_TOL = 1e-4
LM_LOGZ_TOL = 5e-4
LM_TIE_TOL = 5e-4

BASE = synth.WORKLOADS["r128_g16_v151936"]
SMALL = [
    # (R, gamma, V, rank, d, temperatures): every row compared
    (5, 4, 4104, 256, 256, (1.0, 0.7, 0.0)),    # ragged last tile, one partial M-tile
    (130, 3, 8200, 128, 384, (1.0, 0.0)),       # two M-tiles, the second with 2 rows
    (3, 5, 2056, 64, 128, (1.0, 0.0)),          # rank 64, one LM K-chunk
    (64, 2, 151936, 192, 512, (1.0,)),          # the long vocabulary, rank 192
]


def _inputs(wl, rnd):
    W1, W2, _ = synth.weights(wl)
    W_lm = synth.lm_head_weight(wl)
    h = np.stack([synth.hidden(wl, rnd, r) for r in range(wl.R)])
    anchors = synth.anchors(wl, rnd)
    return W1, W2, W_lm, h, anchors


def _gpu_draft(wl, W1, W2, W_lm, h, anchors, temperature, rnd):
    import semi_autoregressive_speculative_gb300 as pkg
    dev = torch.device("cuda", 0)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    hd, Wl, W1d, W2d, ad = t(h.view(np.int16)), t(W_lm.view(np.int16)), t(W1.view(np.int16)), \
        t(W2.view(np.int16)), t(anchors.astype(np.int32))
    tok = torch.empty((wl.R, wl.gamma), dtype=torch.int32, device=dev)
    pd = torch.empty((wl.R, wl.gamma), dtype=torch.float32, device=dev)
    lz = torch.empty_like(pd)
    ws = torch.zeros(pkg.lib().dspark_workspace_size(wl.R, wl.gamma, wl.V, wl.rank, wl.d), dtype=torch.uint8,
                     device=dev)
    pkg.dspark_markov_draft_lmhead(hd, Wl, W1d, W2d, ad, temperature, wl.seed, rnd, tok, pd, lz, ws)
    torch.cuda.synchronize()
    status = int(ws[:4].view(torch.int32).item())
    return host(tok), host(pd), host(lz), status


def _check(wl, h, W_lm, anchors, tok, pd, lz, temperature, rnd, requests):
    """check_draft on the oracle's U = h . W_lm of the compared requests only."""
    req = np.asarray(list(requests))
    rows = oracle.lm_head_logits(h[req], W_lm)  # one pass over W_lm for all compared rows
    inp = types.SimpleNamespace(U=_Rows({int(r): rows[i] for i, r in enumerate(req)}), anchors=anchors)
    counts = {}
    div, ties = check_draft(wl, inp, tok, pd, lz, temperature, rnd, req, counts=counts, cdf_tol=LM_CDF_TOL,
                            logz_tol=LM_LOGZ_TOL, tie_tol=LM_TIE_TOL)
    return div, ties, counts["compared"]


class _Rows:
    """U [R, gamma, V] of which only some requests' rows are formed: indexed
    by a request, an array of requests or (request, position)."""

    def __init__(self, rows):
        self.rows = rows

    def __getitem__(self, key):
        if isinstance(key, tuple):
            return self.rows[int(key[0])][key[1:]]
        if isinstance(key, np.ndarray):
            return np.stack([self.rows[int(k)] for k in key])
        return self.rows[int(key)]


@pytest.mark.gpu
@pytest.mark.parametrize("R,gamma,V,rank,d,temps", SMALL, ids=[f"r{c[0]}_g{c[1]}_v{c[2]}_rank{c[3]}_d{c[4]}"
                                                                for c in SMALL])
def test_lmhead_draft_matches_oracle_every_row(R, gamma, V, rank, d, temps):
    wl = synth.scaled(BASE, R=R, gamma=gamma, V=V, rank=rank, d=d, name=f"lm_r{R}_g{gamma}_v{V}_d{d}")
    rnd = 1
    W1, W2, W_lm, h, anchors = _inputs(wl, rnd)
    for temperature in temps:
        tok, pd, lz, status = _gpu_draft(wl, W1, W2, W_lm, h, anchors, temperature, rnd)
        assert status == 0
        assert np.all((tok >= 0) & (tok < V))
        div, ties, compared = _check(wl, h, W_lm, anchors, tok, pd, lz, temperature, rnd, range(R))
        assert compared >= 0.5 * R * gamma, (compared, R * gamma)
        assert div + ties <= max(1, R // 4), (div, ties)


@pytest.mark.gpu
@pytest.mark.parametrize("temperature", [1.0, 0.0])
def test_lmhead_draft_full_size_batch128(temperature):
    """The batch-128 workload (R=128, gamma=16, V=151936, d=4096) with W_lm
    [4096, 151936] on the device; sampled rows of every tensor-memory lane
    quarter against the oracle."""
    wl = BASE
    rnd = 0
    W1, W2, W_lm, h, anchors = _inputs(wl, rnd)
    tok, pd, lz, status = _gpu_draft(wl, W1, W2, W_lm, h, anchors, temperature, rnd)
    assert status == 0
    assert np.all((tok >= 0) & (tok < wl.V))
    req = sample_requests(wl.R)
    div, ties, compared = _check(wl, h, W_lm, anchors, tok, pd, lz, temperature, rnd, req)
    assert compared >= 0.5 * len(req) * wl.gamma, (compared, len(req) * wl.gamma)
    assert div + ties <= max(1, len(req) // 4), (div, ties)
    if temperature > 0:
        assert np.all(pd > 0.0) and np.all(pd <= 1.0 + PROB_TOL)
