"""The C-ABI library builds, loads, exports every symbol include/dspark.h
declares, and rejects invalid arguments on the host (no GPU needed: each
rejected call returns before touching CUDA)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from semi_autoregressive_speculative_gb300 import build
    build.build()
    import semi_autoregressive_speculative_gb300 as pkg
    return pkg.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "dspark.h")).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t)\s+\*?\s*(dspark_\w+)\s*\(", src, re.M)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert len(names) >= 6
    for n in names:
        assert hasattr(L, n), n
    import semi_autoregressive_speculative_gb300 as pkg
    assert set(names) == set(pkg.EXPORTS)


def test_workspace_size(L):
    s = L.dspark_workspace_size(128, 16, 151936, 256, 4096)
    assert s > 0 and s % 256 == 0
    assert L.dspark_workspace_size(-1, 16, 4096, 256, 64) == 0
    assert L.dspark_workspace_size(4, 65, 4096, 256, 64) == 0
    assert L.dspark_workspace_size(4, 7, 4096, 256, 64) < s


FAKE = 1 << 20  # a 16-byte-aligned non-null address; never dereferenced on rejected calls


def _draft(L, R=4, gamma=7, V=4096, rank=256, T=1.0, U=FAKE, ws=FAKE, wsb=1 << 30, W1=FAKE):
    return L.dspark_markov_draft(U, W1, FAKE, FAKE, R, gamma, V, rank, T, 0, 0, FAKE, FAKE, FAKE, ws, wsb, None)


def test_draft_validation(L):
    assert _draft(L, R=-1) == -1
    assert _draft(L, gamma=0) == -1
    assert _draft(L, T=-1.0) == -1
    assert _draft(L, T=float("nan")) == -1
    assert _draft(L, T=float("inf")) == -1
    assert _draft(L, V=4100) == -2          # V % 8
    assert _draft(L, rank=100) == -2
    assert _draft(L, rank=512) == -2
    assert _draft(L, gamma=65) == -2
    assert _draft(L, U=0) == -1              # null
    assert _draft(L, U=FAKE + 4) == -1       # misaligned
    assert _draft(L, W1=FAKE + 8) == -1
    assert _draft(L, ws=FAKE + 16) == -1     # workspace not 256-aligned
    assert _draft(L, wsb=100) == -1          # workspace too small
    assert _draft(L, R=0) == 0               # empty batch: nothing to do


def _draft_lm(L, R=4, gamma=7, V=4096, rank=256, d=256, T=1.0, h=FAKE, W_lm=FAKE, ws=FAKE, wsb=1 << 30):
    return L.dspark_markov_draft_lmhead(h, W_lm, FAKE, FAKE, FAKE, R, gamma, V, rank, d, T, 0, 0, FAKE, FAKE, FAKE,
                                        ws, wsb, None)


def test_lmhead_draft_validation(L):
    assert _draft_lm(L, d=0) == -1
    assert _draft_lm(L, d=200) == -2         # d % 128
    assert _draft_lm(L, d=65536 + 128) == -2
    assert _draft_lm(L, V=4100) == -2
    assert _draft_lm(L, rank=100) == -2
    assert _draft_lm(L, T=-1.0) == -1
    assert _draft_lm(L, h=0) == -1
    assert _draft_lm(L, W_lm=0) == -1
    assert _draft_lm(L, h=FAKE + 4) == -1    # misaligned
    assert _draft_lm(L, W_lm=FAKE + 8) == -1
    assert _draft_lm(L, ws=FAKE + 16) == -1
    assert _draft_lm(L, wsb=100) == -1
    assert _draft_lm(L, R=0) == 0


def test_schedule_validation(L):
    def call(R=4, gamma=7, sps_len=4 * 8 + 1, mode=0, a=FAKE):
        return L.dspark_schedule(a, R, gamma, FAKE, sps_len, mode, 0, FAKE, FAKE, FAKE, FAKE, FAKE, 4, None)
    assert call(sps_len=32) == -1
    assert call(mode=3) == -1
    assert call(R=0) == -1
    assert call(R=1025, gamma=8, sps_len=1025 * 9 + 1) == -2   # R * gamma > 8192
    assert call(a=0) == -1


def test_confidence_and_verify_validation(L):
    def conf(h=FAKE, R=4, d=64, sts=None):
        return L.dspark_confidence(h, FAKE, FAKE, sts, FAKE, FAKE, R, 7, d, 256, 4096, FAKE, FAKE, FAKE, 4, None)
    assert conf(d=0) == -1
    assert conf(h=0) == -1
    assert conf(R=0) == 0
    assert conf(R=0, sts=FAKE) == 0

    def verify(T=FAKE, V=4096, temp=1.0, wsb=1 << 30):
        return L.dspark_verify(T, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 7, V, 256, temp, 0, 0,
                               FAKE, FAKE, None, FAKE, wsb, None)
    assert verify(T=0) == -1
    assert verify(T=FAKE + 4) == -1
    assert verify(V=12) == -2
    assert verify(temp=-0.5) == -1
    assert verify(wsb=8) == -1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import semi_autoregressive_speculative_gb300 as pkg
    monkeypatch.setattr(pkg, "_lib", None)
    monkeypatch.setattr(pkg, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        pkg.lib()


def test_load_rows_validation(L):
    def call(T_host=FAKE, lens=FAKE, R=4, gamma=7, V=4096, T=FAKE, ws=FAKE):
        return L.dspark_load_verified_rows(T_host, lens, R, gamma, V, T, ws, None)
    assert call(R=-1) == -1
    assert call(gamma=0) == -1
    assert call(V=4) == -1
    assert call(V=4100) == -2          # V % 8
    assert call(gamma=65) == -2
    assert call(T_host=0) == -1
    assert call(lens=0) == -1
    assert call(T=0) == -1
    assert call(ws=0) == -1
    assert call(T_host=FAKE + 4) == -1  # misaligned
    assert call(T=FAKE + 8) == -1
    assert call(ws=FAKE + 16) == -1     # workspace not 256-aligned
    assert call(R=0) == 0               # empty batch: nothing to do


def test_load_rows_binding_checks_the_host_shape():
    # the binding's own shape check runs before the library is called
    import torch
    import semi_autoregressive_speculative_gb300 as pkg
    T = torch.empty((3, 5, 16))
    with pytest.raises(ValueError):
        pkg.dspark_load_verified_rows(torch.empty((3, 4, 16)), None, T, None)
