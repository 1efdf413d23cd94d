"""Pins of the oracle's counter-based uniforms.

Philox4x64-10 is pinned to the known-answer vectors published with its
definition (tests/golden/philox4x64_10_kat.txt) and to numpy's independent
implementation, numpy.random.Philox.
"""
import os

import numpy as np
from scipy import stats

GOLD = os.path.join(os.path.dirname(__file__), "golden", "philox4x64_10_kat.txt")
MASK64 = (1 << 64) - 1


def _kat():
    rows = []
    with open(GOLD) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            v = [int(x, 16) for x in line.split()]
            rows.append((v[0:4], v[4:6], v[6:10]))
    return rows


def test_known_answer_vectors(orc):
    rows = _kat()
    assert len(rows) == 3
    for ctr, key, out in rows:
        assert [int(x) for x in orc.philox4x64_10(ctr, key)] == out


def _numpy_block(ctr, key):
    # numpy's Philox steps its 256-bit counter (word 0 least significant)
    # before producing a block, so counter c is produced from state c - 1.
    c = sum(int(w) << (64 * i) for i, w in enumerate(ctr))
    c = (c - 1) % (1 << 256)
    state = [(c >> (64 * i)) & MASK64 for i in range(4)]
    bg = np.random.Philox(counter=np.array(state, np.uint64), key=np.array(key, np.uint64))
    return [int(x) for x in bg.random_raw(4)]


def test_matches_numpy_philox(orc):
    rng = np.random.default_rng(123)
    cases = [[0, 0, 0, 0], [1, 2, 3, 4], [7, 1 << 63, 5, 2], [0, 1, 0, 0]]
    cases += [[int(x) for x in rng.integers(0, 1 << 63, 4)] for _ in range(40)]
    for ctr in cases:
        for key in ([0, 0], [5, 0], [MASK64, 3]):
            assert [int(x) for x in orc.philox4x64_10(ctr, key)] == _numpy_block(ctr, key)


def test_uniform_is_top_24_bits_of_word0(orc):
    for seed, rnd, req, pos, pur in [(0, 0, 0, 0, 0), (1, 3, 17, 5, 2), (4, 7, 255, 15, 1)]:
        out = orc.philox4x64_10([rnd, req, pos, pur], [seed, 0])
        u = orc.uniform(seed, rnd, req, pos, pur)
        assert u == (int(out[0]) >> 40) / 2**24
        assert 0.0 <= u < 1.0
        assert np.float32(u) == u  # exactly representable in binary32


def test_uniform_distribution_and_stream_independence(orc):
    n = 20000
    us = np.array([orc.uniform(9, 0, r, 0, 0) for r in range(n)])
    assert stats.kstest(us, "uniform").pvalue > 1e-4
    vs = np.array([orc.uniform(9, 0, r, 0, 1) for r in range(n)])
    assert abs(np.corrcoef(us, vs)[0, 1]) < 4 / np.sqrt(n)
