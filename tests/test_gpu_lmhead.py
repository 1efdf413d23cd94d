"""The fused LM-head draft (dspark_markov_draft_lmhead) against the oracle.

The oracle forms U = h . W_lm (oracle.lm_head_logits: fp64 sums rounded once
to fp32) and drafts from it exactly as for a given U.  The kernel instead sums
the d LM-head products and the rank bias products of a logit in one fp32
tensor-core accumulator, K = 16 products per MMA step, (d + rank) / 16 steps
in all.  Allowing each step to lose one fp32 unit in the last place of a
logit of magnitude up to 32 bounds the kernel's logit error by

    E = (d + rank) / 16 * 2^-23 * 32        (1.0e-3 at d = 4096, 1.8e-3 at d = 7168)

and the comparison allows E on log Z, 2E on a greedy top-two gap, on the CDF
and on p_d (|dp| <= p (1 - p) * 2E), never less than the U-path draft's own
tolerances.  Measured: about 7e-4 on the logits at d = 7168.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import CDF_TOL, LOGZ_TOL, PROB_TOL, check_draft_forced, host, sample_requests
from semi_autoregressive_speculative_gb300 import synth


def lm_tolerances(wl):
    E = (wl.d + wl.rank) / 16 * 2.0 ** -23 * 32.0
    return dict(cdf_tol=max(CDF_TOL, 2 * E), logz_tol=max(LOGZ_TOL, E), tie_tol=max(1e-4, 2 * E),
                prob_tol=max(PROB_TOL, 2 * E))


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
    """Every position of the compared requests against the oracle drafting
    from its U = h . W_lm, conditioned on the kernel's own previous tokens."""
    req = [int(r) for r in requests]
    rows = oracle.lm_head_logits(h[req], W_lm)  # one pass over W_lm for all compared rows
    U_rows = {r: rows[i] for i, r in enumerate(req)}
    return check_draft_forced(wl, U_rows, anchors, tok, pd, lz, temperature, rnd, req, **lm_tolerances(wl))


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
        differ = _check(wl, h, W_lm, anchors, tok, pd, lz, temperature, rnd, range(R))
        assert differ <= max(1, R * gamma // 10), differ


FULL = [("r128_g16_v151936", 1.0), ("r128_g16_v151936", 0.0), ("r256_g16_v129280_d7168", 1.0)]


@pytest.mark.gpu
@pytest.mark.parametrize("name,temperature", FULL, ids=[f"{n}_T{t}" for n, t in FULL])
def test_lmhead_draft_full_size(name, temperature):
    """Full size with W_lm on the device: the batch-128 workload (R=128,
    gamma=16, V=151936, d=4096; W_lm 1.25 GB) and the two-M-tile workload
    (R=256, V=129280, d=7168; W_lm 1.85 GB); sampled rows of every
    tensor-memory lane quarter of every M-tile against the oracle."""
    wl = synth.WORKLOADS[name]
    rnd = 0
    W1, W2, W_lm, h, anchors = _inputs(wl, rnd)
    tok, pd, lz, status = _gpu_draft(wl, W1, W2, W_lm, h, anchors, temperature, rnd)
    assert status == 0
    assert np.all((tok >= 0) & (tok < wl.V))
    req = sample_requests(wl.R)
    differ = _check(wl, h, W_lm, anchors, tok, pd, lz, temperature, rnd, req)
    # every differing draw was checked to lie within the CDF tolerance; at these
    # vocabularies about one draw in ten lands that close to a boundary
    assert differ <= len(req) * wl.gamma // 4, differ
    if temperature > 0:
        assert np.all(pd > 0.0) and np.all(pd <= 1.0 + lm_tolerances(wl)["prob_tol"])
