"""Whole rounds on the GPU: the chained device round (draft -> confidence ->
schedule -> verify, several rounds with anchors carried over and the lagged
Top-K budget) against the oracle's own chained round on the same seeded
inputs, plus CUDA-graph capture of a round."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import CDF_TOL, check_verify, device_round, host, weights
from semi_autoregressive_speculative_gb300 import synth
from semi_autoregressive_speculative_gb300.round import MODE_EARLY_STOP, MODE_TOP_K

pytestmark = pytest.mark.gpu


def _target(wl, inp, tokens, rnd):
    """T = U + Markov bias of the drafted prefix + noise (oracle bias)."""
    W1, W2, _ = weights(wl)
    T = np.empty((wl.R, wl.gamma + 1, wl.V), np.float32)
    for r in range(wl.R):
        prevs = [int(inp.anchors[r])] + [int(x) for x in tokens[r, :-1]]
        bias = np.stack([oracle.markov_bias(W1, W2, pv) for pv in prevs])
        T[r] = synth.compose_target(inp.U[r], bias, synth.target_noise(wl, rnd, r), synth.bonus_base(wl, rnd, r))
    return T


def _oracle_round(wl, inp, sps, mode, K, temperature, rnd):
    W1, W2, w = weights(wl)
    tok, pd, lz = oracle.draft(inp.U, W1, W2, inp.anchors, temperature, wl.seed, rnd)
    c, a = oracle.confidence(inp.h, W1, w, inp.anchors, tok)
    s = oracle.schedule(a, sps, mode, K)
    T = _target(wl, inp, tok, rnd)
    na, nx = oracle.verify(T, inp.U, W1, W2, inp.anchors, tok, s["lens"], temperature, wl.seed, rnd)
    return dict(tok=tok, pd=pd, c=c, a=a, sched=s, T=T, na=na, nx=nx)


def _staircase_scaled(wl):
    # the staircase with its cliffs scaled to this batch: B_max / 8, / 4, / 2
    B = np.arange(wl.B_max + 1, dtype=np.float64)
    q = wl.B_max / 8
    return 1000.0 / (1.0 + 0.25 * (B >= q) + 0.5 * (B >= 2 * q) + 1.0 * (B >= 4 * q))


@pytest.mark.parametrize("temperature", [1.0, 0.0])
def test_chained_rounds_lagged_top_k(temperature):
    base = synth.WORKLOADS["r512_g16_v32768_staircase"]
    wl = synth.scaled(base, R=12, gamma=6, V=2048, d=64, name="chain_r12")
    sps = _staircase_scaled(wl)
    anchors = synth.anchors(wl, 0)
    history = []
    for rnd in range(4):
        inp = synth.round_inputs(wl, rnd, anchor_override=anchors)
        mode = MODE_TOP_K
        K = wl.R * wl.gamma if len(history) < 2 else history[-2]
        orc = _oracle_round(wl, inp, sps, mode, K, temperature, rnd)
        dr, _ = device_round(wl, inp)
        dr.sps.copy_(torch.from_numpy(sps))
        dr.draft(temperature, wl.seed, rnd)
        dr.confidence()
        dr.schedule(mode, K)
        tok_g = host(dr.tokens)
        if not np.array_equal(tok_g, orc["tok"]):
            # only a sampled draw within CDF_TOL of a boundary may differ; the
            # chains then legitimately part ways
            assert temperature > 0
            r, j = [int(v[0]) for v in np.nonzero(tok_g != orc["tok"])]
            W1, W2, _ = weights(wl)
            prev = int(inp.anchors[r]) if j == 0 else int(orc["tok"][r, j - 1])
            p, _ = oracle.draft_probs(inp.U[r, j], W1, W2, prev, temperature)
            cdf = np.cumsum(p)
            u = oracle.uniform(wl.seed, rnd, r, j, 0)
            x = int(tok_g[r, j])
            assert (cdf[x - 1] if x else 0.0) - CDF_TOL <= u < cdf[x] + CDF_TOL
            return
        assert np.max(np.abs(host(dr.c) - orc["c"])) <= 1e-4
        lens_g = host(dr.lens)
        if not np.array_equal(lens_g, orc["sched"]["lens"]):
            # the device's own confidences differ from the oracle's within
            # 1e-4 and may flip a near tie in the ranking; fed the oracle's a,
            # the device scheduler must agree bit for bit
            dr.a.copy_(torch.from_numpy(orc["a"]))
            dr.schedule(mode, K)
            lens_g = host(dr.lens)
        assert np.array_equal(lens_g, orc["sched"]["lens"])
        assert int(dr.sched_out[0]) == orc["sched"]["total_b"]
        history.append(int(dr.sched_out[1]))
        assert history[-1] == orc["sched"]["argmax_b"]
        dr.T.copy_(torch.from_numpy(orc["T"]))
        dr.verify(temperature, wl.seed, rnd)
        na, nx = host(dr.n_accept), host(dr.next_token)
        # every request against the oracle: bit-exact, except a decision within
        # 1e-5 of its threshold (check_verify's exemptions)
        ex = check_verify(wl, inp, orc["T"], orc["tok"], orc["sched"]["lens"], na, nx, temperature, rnd,
                          range(wl.R))
        if temperature == 0.0:
            assert ex == 0
        if ex:
            return  # the chains part ways: later rounds would start from other anchors
        assert np.array_equal(na, orc["na"]) and np.array_equal(nx, orc["nx"])
        anchors = orc["nx"]
        assert dr.status() == 0


def test_round_in_cuda_graph():
    wl = synth.scaled(synth.WORKLOADS["tiny_r4_g7_v4096"], R=8, gamma=5, V=4096, d=64, name="graph")
    dr, inp = device_round(wl)
    W1, W2, _ = weights(wl)
    T = _target(wl, inp, np.zeros((wl.R, wl.gamma), np.int32), 0)
    dr.T.copy_(torch.from_numpy(T))

    def run():
        dr.draft(1.0, wl.seed, 0)
        dr.confidence()
        dr.schedule(MODE_EARLY_STOP)
        dr.verify(1.0, wl.seed, 0)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run()  # warm-up outside capture (sets kernel attributes)
    torch.cuda.synchronize()
    eager = [host(x).copy() for x in (dr.tokens, dr.lens, dr.n_accept, dr.next_token)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run()
    dr.tokens.zero_()
    dr.next_token.zero_()
    g.replay()
    torch.cuda.synchronize()
    replay = [host(x) for x in (dr.tokens, dr.lens, dr.n_accept, dr.next_token)]
    for e, r in zip(eager, replay):
        assert np.array_equal(e, r)
    assert dr.status() == 0


def test_status_flags_bad_anchor():
    wl = synth.scaled(synth.WORKLOADS["tiny_r4_g7_v4096"], R=4, gamma=2, V=512, d=16, name="badanchor")
    dr, inp = device_round(wl)
    dr.anchors[1] = wl.V + 5  # out of range: clamped to 0 and reported
    dr.draft(1.0, 0, 0)
    tok = host(dr.tokens)
    assert tok.min() >= 0 and tok.max() < wl.V
    from semi_autoregressive_speculative_gb300 import DSPARK_STATUS_BAD_TOKEN
    assert dr.status() & DSPARK_STATUS_BAD_TOKEN
    dr.clear_status()
    assert dr.status() == 0
    # greedy: the bad row drafts exactly as with anchor 0, the others as given
    dr.draft(0.0, 0, 0)
    tok = host(dr.tokens)
    W1, W2, _ = weights(wl)
    anchors = np.array(inp.anchors, np.int32)
    anchors[1] = 0
    tok_o, _, _ = oracle.draft(inp.U, W1, W2, anchors, 0.0, 0, 0)
    assert np.array_equal(tok, tok_o), (tok, tok_o)
    assert dr.status() & DSPARK_STATUS_BAD_TOKEN


def test_nonfinite_logits_reported():
    wl = synth.scaled(synth.WORKLOADS["tiny_r4_g7_v4096"], R=2, gamma=2, V=512, d=16, name="nan")
    dr, inp = device_round(wl)
    dr.U[0, 0, 7] = float("nan")
    dr.draft(1.0, 0, 0)
    torch.cuda.synchronize()
    from semi_autoregressive_speculative_gb300 import DSPARK_STATUS_NONFINITE
    assert dr.status() & DSPARK_STATUS_NONFINITE
    tok = host(dr.tokens)
    assert tok.min() >= 0 and tok.max() < wl.V


def test_bounded_wait_gives_up_and_reports_timeout():
    # a device wait on a phase that nothing completes gives up after its limit,
    # reports DSPARK_STATUS_TIMEOUT and returns: the context stays usable
    from semi_autoregressive_speculative_gb300 import DSPARK_STATUS_TIMEOUT, dspark_selftest_bounded_wait
    wl = synth.scaled(synth.WORKLOADS["tiny_r4_g7_v4096"], R=4, gamma=3, V=512, d=16, name="timeout")
    dr, inp = device_round(wl)
    dspark_selftest_bounded_wait(dr.workspace)
    torch.cuda.synchronize()
    assert dr.status() & DSPARK_STATUS_TIMEOUT
    dr.clear_status()
    dr.draft(1.0, wl.seed, 0)
    tok = host(dr.tokens)
    assert tok.min() >= 0 and tok.max() < wl.V
    assert dr.status() == 0


def test_one_graph_many_rounds_device_decided_lengths():
    # One captured round replayed on new inputs: the scheduler decides each
    # request's verify length on the device, and verify consumes those
    # variable lengths inside the same graph; no length is baked into it.
    # Every replay is checked against the eager run and against the oracle's
    # round on the same inputs.
    wl = synth.scaled(synth.WORKLOADS["tiny_r4_g7_v4096"], R=16, gamma=6, V=4096, d=64, name="graph_lens")
    dr, _ = device_round(wl)
    # a throughput curve with cliffs inside this batch, so that early stop
    # admits a different set of positions for different confidences
    sps = _staircase_scaled(wl)
    dr.sps.copy_(torch.from_numpy(sps))
    W1, W2, w = weights(wl)
    loaded = {}

    def load(rnd):
        inp = synth.round_inputs(wl, rnd)
        T = _target(wl, inp, np.zeros((wl.R, wl.gamma), np.int32), rnd)
        dr.set_round(inp.U, inp.h, inp.anchors)
        dr.T.copy_(torch.from_numpy(T))
        loaded[rnd] = (inp, T)

    def oracle_round(rnd):
        # the captured calls use Philox round 0 on every input set
        inp, T = loaded[rnd]
        tok, _, _ = oracle.draft(inp.U, W1, W2, inp.anchors, 1.0, wl.seed, 0)
        _, a = oracle.confidence(inp.h, W1, w, inp.anchors, tok)
        sch = oracle.schedule(a, sps, MODE_EARLY_STOP)
        return inp, T, tok, a, sch

    def run():
        dr.draft(1.0, wl.seed, 0)
        dr.confidence()
        dr.schedule(MODE_EARLY_STOP)
        dr.verify(1.0, wl.seed, 0)

    outs = (dr.tokens, dr.a, dr.lens, dr.sched_out, dr.n_accept, dr.next_token)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    load(0)
    with torch.cuda.stream(s):
        run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run()
    lens_seen = []
    for rnd in range(3):
        load(rnd)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            run()
        torch.cuda.synchronize()
        eager = [host(x).copy() for x in outs]
        for x in outs:
            x.zero_()
        load(rnd)
        g.replay()
        torch.cuda.synchronize()
        replay = [host(x) for x in outs]
        for e, r in zip(eager, replay):
            assert np.array_equal(e, r)
        lens_seen.append(tuple(replay[2][: wl.R]))
        assert int(replay[3][0]) == int(np.sum(replay[2][: wl.R]))
        assert np.all(replay[4][: wl.R] <= replay[2][: wl.R])
        # the replay against the oracle's round on the same inputs
        inp, T, tok_o, a_o, sch = oracle_round(rnd)
        tok_g = replay[0]
        if not np.array_equal(tok_g, tok_o):
            # only a draw within 1e-5 of a CDF boundary may differ; the rest of
            # that round then conditions on another prefix and is not compared
            r, j = [int(v[0]) for v in np.nonzero(tok_g != tok_o)]
            prev = int(inp.anchors[r]) if j == 0 else int(tok_o[r, j - 1])
            p, _ = oracle.draft_probs(inp.U[r, j], W1, W2, prev, 1.0)
            cdf = np.cumsum(p)
            u = oracle.uniform(wl.seed, 0, r, j, 0)
            x = int(tok_g[r, j])
            assert (cdf[x - 1] if x else 0.0) - CDF_TOL <= u < cdf[x] + CDF_TOL
            continue
        assert np.max(np.abs(replay[1] - a_o)) <= 1e-4
        assert np.array_equal(replay[2], sch["lens"]) and int(replay[3][0]) == sch["total_b"]
        check_verify(wl, inp, T, tok_o, sch["lens"], replay[4], replay[5], 1.0, 0, range(wl.R))
    assert len(set(lens_seen)) > 1  # the lengths really are decided per replay
    assert dr.status() == 0
