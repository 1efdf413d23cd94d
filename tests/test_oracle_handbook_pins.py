"""Pins of the oracle against the printed outputs of the page
"投机解码的新做法：整块草稿、按负载验证与 PD 分离":

* its H100 cost-model table (section "负载越高，K 越要小"),
* its adaptive-verification planner (section "按负载决定验证多少"), reproduced by
  the oracle's scheduler fed the page's confidence matrices,
* its Markov-chain toy (section "一次前向给出一整块草稿"), reproduced by the
  oracle's greedy Markov draft with U = 0 and W1 W2 = log P.

The page's inputs come from torch's CPU generator with seed 0; the recipes
below draw the same numbers in the same order.
"""
import os

import numpy as np
import pytest

from oracle import cost_model
from semi_autoregressive_speculative_gb300 import synth

torch = pytest.importorskip("torch")
GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            out.append(line.split())
    return out


def test_cost_model_table():
    for batch, none, kseq, sseq, kblk, sblk in _rows("handbook_cost_model.txt"):
        batch = int(batch)
        base = cost_model.tokens_per_second(batch, 0, False)
        assert f"{base:.0f}" == none
        ks = cost_model.best_k(batch, one_shot_draft=False)
        kb = cost_model.best_k(batch, one_shot_draft=True)
        assert ks == int(kseq) and kb == int(kblk)
        assert f"{cost_model.tokens_per_second(batch, ks, False) / base:.2f}" == sseq
        assert f"{cost_model.tokens_per_second(batch, kb, True) / base:.2f}" == sblk


def test_workload_sps_tables_follow_cost_model():
    for name in ("tiny_r4_g7_v4096", "r128_g16_v151936"):
        wl = synth.WORKLOADS[name]
        tab = synth.sps_table(wl)
        ref = np.array([cost_model.sps_target_only(B) for B in range(wl.B_max + 1)])
        np.testing.assert_allclose(tab, ref, rtol=1e-15, atol=0)


def _planner_confidences():
    torch.manual_seed(0)
    K = 7
    out = {}
    for batch in (16, 128, 512):
        good = batch // 2
        level = torch.cat([torch.full((good, K), 0.9), torch.full((batch - good, K), 0.55)])
        jitter = torch.rand(batch, K).mul(0.2).add(0.9)
        out[batch] = (level * jitter).clamp(max=0.99).numpy().astype(np.float32)
    return out


def test_adaptive_planner(orc):
    confs = _planner_confidences()
    for batch, admitted, kept_good, kept_poor, none, fixed, adaptive in _rows(
            "handbook_adaptive_planner.txt"):
        batch = int(batch)
        conf = confs[batch]
        R, K = conf.shape
        a = orc.survival(conf)
        assert np.all(np.diff(a, axis=1) <= 0)
        sps = np.array([cost_model.sps_with_draft(B) for B in range(R * (1 + K) + 1)])
        # the page's planner is a global argmax over the budget; early stop
        # reaches the same budget on these unimodal curves
        res_es = orc.schedule(a, sps, orc.MODE_EARLY_STOP)
        assert res_es["argmax_b"] == int(admitted)
        assert res_es["total_b"] == int(admitted)
        res_k = orc.schedule(a, sps, orc.MODE_TOP_K, res_es["argmax_b"])
        assert res_k["total_b"] == int(admitted)
        assert f"{res_es['theta']:.0f}" == adaptive
        lens = res_es["lens"]
        assert lens.sum() == int(admitted)
        assert f"{lens[:batch // 2].mean():.1f}" == kept_good
        assert f"{lens[batch // 2:].mean():.1f}" == kept_poor
        verify_all = (batch + a.astype(np.float64).sum()) * cost_model.sps_with_draft(batch * (1 + K))
        assert f"{verify_all:.0f}" == fixed
        assert f"{batch * cost_model.sps_target_only(batch):.0f}" == none


def _handbook_chain():
    torch.manual_seed(0)
    V = 64
    P = torch.full((V, V), 0.1 / (V - 2))
    for src in range(V):
        b, c = torch.randperm(V)[:2]
        P[src, b], P[src, c] = 0.45, 0.45
    return P.numpy()


def _expected_accepted(P, draft, last):
    total, run, prev = 0.0, 1.0, last
    for x in draft:
        run *= float(P[prev, x])
        total += run
        prev = x
    return total


def test_markov_toy(orc):
    (indep, markov), = _rows("handbook_markov_toy.txt")
    P = _handbook_chain()
    V, K = P.shape[0], 6
    # independent positions: the argmax of each marginal i steps ahead.  The
    # marginals hold exact ties, so this baseline is taken with torch's own
    # float32 product and first-maximum argmax, as on the page.
    Pt = torch.from_numpy(P)
    par = 0.0
    for t in range(V):
        dist = torch.zeros(V)
        dist[t] = 1
        draft = []
        for _ in range(K):
            dist = dist @ Pt
            draft.append(int(dist.argmax()))
        par += _expected_accepted(P, draft, t)
    assert f"{par / V:.2f}" == indep
    # the oracle's greedy Markov draft with U = 0 and W1 W2 = log P
    W1 = synth.to_bf16_bits(np.log(P))           # [V, r = V]
    W2 = synth.to_bf16_bits(np.eye(V, dtype=np.float32))  # [r = V, V]
    U = np.zeros((V, K, V), np.float32)
    tokens, _, _ = orc.draft(U, W1, W2, np.arange(V, dtype=np.int32), 0.0, seed=0, rnd=0)
    mar = sum(_expected_accepted(P, tokens[t], t) for t in range(V)) / V
    assert f"{mar:.2f}" == markov
