"""dspark_markov_draft_noalloc against dspark_markov_draft.

The no-alloc entry point serves callers that cannot obtain device memory where
they draft.  Examples are an engine capturing its decode step into a CUDA
graph, a serving loop that bans allocator calls because they can synchronise
the device, and a plug-in without an allocator.  It keeps its scratch in the
library's own fixed 16 MiB device array instead of a caller workspace.

Its results must be those of the workspace entry point on the same inputs,
call after call: the array is shared and keeps the previous call's contents.
This file sorts last so that a stop-at-first-failure run has run every other
test before it.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import LOGZ_TOL, PROB_TOL, device_round, host
from semi_autoregressive_speculative_gb300 import synth

FAKE = 1 << 20  # a 16-byte-aligned non-null address; never dereferenced on rejected calls


def test_rejects_shapes_beyond_the_static_scratch():
    import semi_autoregressive_speculative_gb300 as pkg
    from semi_autoregressive_speculative_gb300 import build
    build.build()
    L = pkg.lib()
    # R = 1024 at V = 151936 needs about 45 MiB of partials: rejected before any CUDA call
    rc = L.dspark_markov_draft_noalloc(FAKE, FAKE, FAKE, FAKE, 1024, 16, 151936, 256, 1.0, 0, 0, FAKE, FAKE, FAKE,
                                       None, None)
    assert rc == pkg.DSPARK_ERR_STATIC_SCRATCH_TOO_SMALL
    # the usual argument rules still apply first
    assert L.dspark_markov_draft_noalloc(FAKE, FAKE, FAKE, FAKE, 4, 7, 4100, 256, 1.0, 0, 0, FAKE, FAKE, FAKE,
                                         None, None) == pkg.DSPARK_ERR_UNSUPPORTED_SHAPE
    assert L.dspark_markov_draft_noalloc(0, FAKE, FAKE, FAKE, 4, 7, 4096, 256, 1.0, 0, 0, FAKE, FAKE, FAKE,
                                         None, None) == pkg.DSPARK_ERR_INVALID_ARG


def _compare(dr, ref, tok, pd, lz):
    assert np.array_equal(host(tok), ref[0])
    assert np.max(np.abs(host(pd) - ref[1])) <= PROB_TOL
    assert np.all(np.abs(host(lz) - ref[2]) <= LOGZ_TOL * np.maximum(1.0, np.abs(ref[2])))


CASES = [
    # (name, R, gamma, V, temperature)
    ("small_ragged", 5, 4, 4104, 1.0),
    ("two_mtiles_greedy", 130, 3, 8200, 0.0),
    ("batch128_long_vocab", 128, 2, 151936, 1.0),
]


@pytest.mark.gpu
@pytest.mark.parametrize("name,R,gamma,V,temperature", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_workspace_draft_two_calls_in_a_row(name, R, gamma, V, temperature):
    from semi_autoregressive_speculative_gb300 import dspark_markov_draft_noalloc
    wl = synth.scaled(synth.WORKLOADS["r128_g16_v151936"], R=R, gamma=gamma, V=V, d=16, name="noalloc_" + name)
    dr, _ = device_round(wl)
    tok = torch.empty_like(dr.tokens)
    pd = torch.empty_like(dr.pd)
    lz = torch.empty_like(dr.logZ)
    status = torch.full((1,), -1, dtype=torch.int32, device=dr.device)
    for rnd in (0, 1):
        # the workspace entry point on these inputs
        dr.draft(temperature, wl.seed, rnd)
        ref = (host(dr.tokens).copy(), host(dr.pd).copy(), host(dr.logZ).copy())
        assert dr.status() == 0
        # two no-alloc calls in a row, each checked on its own
        for _ in range(2):
            tok.fill_(-7)
            pd.fill_(-1.0)
            lz.fill_(float("nan"))
            dspark_markov_draft_noalloc(dr.U, dr.W1, dr.W2, dr.anchors, temperature, wl.seed, rnd, tok, pd, lz,
                                        status=status)
            torch.cuda.synchronize()
            _compare(dr, ref, tok, pd, lz)
            assert int(status.item()) == 0


def _noalloc_outputs(dr):
    return torch.empty_like(dr.tokens), torch.empty_like(dr.pd), torch.empty_like(dr.logZ)


@pytest.mark.gpu
def test_noalloc_large_shape_then_small_shape():
    """The shared scratch keeps a larger call's partials and sync words; a
    smaller call after it must not read any of them."""
    from semi_autoregressive_speculative_gb300 import dspark_markov_draft_noalloc
    base = synth.WORKLOADS["r128_g16_v151936"]
    shapes = [("large", 256, 2, 129280, 1.0), ("small", 5, 4, 4104, 1.0), ("small_greedy", 130, 3, 8200, 0.0)]
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for name, R, gamma, V, temperature in shapes:
        wl = synth.scaled(base, R=R, gamma=gamma, V=V, d=16, name="noalloc_seq_" + name)
        dr, _ = device_round(wl)
        dr.draft(temperature, wl.seed, 0)
        ref = (host(dr.tokens).copy(), host(dr.pd).copy(), host(dr.logZ).copy())
        assert dr.status() == 0
        tok, pd, lz = _noalloc_outputs(dr)
        dspark_markov_draft_noalloc(dr.U, dr.W1, dr.W2, dr.anchors, temperature, wl.seed, 0, tok, pd, lz,
                                    status=status)
        torch.cuda.synchronize()
        _compare(dr, ref, tok, pd, lz)
        assert int(status.item()) == 0
        del dr
        torch.cuda.empty_cache()


@pytest.mark.gpu
@pytest.mark.parametrize("temperature", [1.0, 0.0])
def test_noalloc_captured_in_a_graph_after_warm_up(temperature):
    """The use the header names: one eager call, then the call recorded into a
    CUDA graph and replayed on new U (written into the same buffer), each replay
    checked against the workspace entry point on that round's inputs."""
    from semi_autoregressive_speculative_gb300 import dspark_markov_draft_noalloc
    wl = synth.scaled(synth.WORKLOADS["r128_g16_v151936"], R=130, gamma=3, V=8200, d=16, name="noalloc_graph")
    dr, _ = device_round(wl)
    tok, pd, lz = _noalloc_outputs(dr)
    status = torch.full((1,), -1, dtype=torch.int32, device=dr.device)
    rnd = 0
    dspark_markov_draft_noalloc(dr.U, dr.W1, dr.W2, dr.anchors, temperature, wl.seed, rnd, tok, pd, lz, status=status)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=side):
        dspark_markov_draft_noalloc(dr.U, dr.W1, dr.W2, dr.anchors, temperature, wl.seed, rnd, tok, pd, lz,
                                    status=status)
    torch.cuda.synchronize()
    for k in range(3):
        # a new round's U in the captured buffer (same seed and round: only U differs)
        inp = synth.round_inputs(wl, k + 1)
        dr.U.copy_(torch.from_numpy(inp.U))
        dr.draft(temperature, wl.seed, rnd)
        ref = (host(dr.tokens).copy(), host(dr.pd).copy(), host(dr.logZ).copy())
        assert dr.status() == 0
        tok.fill_(-7)
        pd.fill_(-1.0)
        lz.fill_(float("nan"))
        status.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        _compare(dr, ref, tok, pd, lz)
        assert int(status.item()) == 0
