"""dspark_load_verified_rows: the admitted target rows copied from page-locked
host memory, bit for bit, and nothing else written.

This is data movement, so the check is its definition: after the call, row j
of request r on the device equals row j of the host tensor for every
j <= lens[r] (lengths clamped to [0, gamma]) and still holds its previous
contents for every other j."""
import numpy as np
import pytest
import torch

SENTINEL = -12345.0


def _run(R, gamma, V, lens, seed=0):
    import semi_autoregressive_speculative_gb300 as pkg
    dev = torch.device("cuda", 0)
    g = torch.Generator().manual_seed(seed)
    T_host = torch.randint(-(1 << 30), 1 << 30, (R, gamma + 1, V), generator=g, dtype=torch.int32)
    T_host = T_host.view(torch.float32).pin_memory()
    T = torch.full((R, gamma + 1, V), SENTINEL, dtype=torch.float32, device=dev)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    pkg.dspark_load_verified_rows(T_host, lens_d, T, ws)
    torch.cuda.synchronize()
    status = int(ws[:4].view(torch.int32).item())
    return T_host, T.cpu(), status


def _check(T_host, T, lens, gamma):
    src = T_host.view(torch.int32)
    out = T.view(torch.int32)
    sentinel = torch.tensor([SENTINEL], dtype=torch.float32).view(torch.int32)
    for r, l in enumerate(lens):
        n = min(max(int(l), 0), gamma) + 1
        assert torch.equal(out[r, :n], src[r, :n]), r
        assert torch.all(out[r, n:] == sentinel), r


CASES = [
    # (R, gamma, V): one partial piece per row; several pieces and a ragged last
    # piece; the batch-128 round's full size
    (5, 4, 4104),
    (37, 7, 70000),
    (128, 16, 151936),
]


@pytest.mark.gpu
@pytest.mark.parametrize("R,gamma,V", CASES, ids=[f"r{c[0]}_g{c[1]}_v{c[2]}" for c in CASES])
def test_load_rows_copies_exactly_the_admitted_rows(R, gamma, V):
    rng = np.random.default_rng(R * 1000 + gamma)
    lens = rng.integers(0, gamma + 1, size=R)
    lens[0], lens[-1] = 0, gamma  # the two extremes
    T_host, T, status = _run(R, gamma, V, lens.tolist())
    assert status == 0
    _check(T_host, T, lens, gamma)


@pytest.mark.gpu
def test_load_rows_clamps_bad_lengths():
    R, gamma, V = 4, 5, 2056
    lens = [-3, gamma + 2, 1, 1 << 30]
    T_host, T, status = _run(R, gamma, V, lens)
    assert status & 8  # DSPARK_STATUS_BAD_LENGTH
    _check(T_host, T, lens, gamma)


@pytest.mark.gpu
def test_load_rows_refuses_memory_that_is_not_pinned_host_memory():
    import semi_autoregressive_speculative_gb300 as pkg
    dev = torch.device("cuda", 0)
    R, gamma, V = 2, 3, 1024
    T = torch.full((R, gamma + 1, V), SENTINEL, device=dev)
    lens = torch.ones(R, dtype=torch.int32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    for src in (torch.zeros(R, gamma + 1, V),                 # pageable host memory
                torch.zeros(R, gamma + 1, V, device=dev)):    # device memory
        with pytest.raises(pkg.DsparkError) as e:
            pkg.dspark_load_verified_rows(src, lens, T, ws)
        assert e.value.code == -1
    torch.cuda.synchronize()
    assert torch.all(T == SENTINEL)
