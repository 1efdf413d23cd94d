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
