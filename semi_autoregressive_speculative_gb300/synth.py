"""Seeded synthetic inputs for one DSpark round.

This module draws random numbers and lays them out; it holds none of the
method's arithmetic (no bias, softmax, confidence, schedule or verify step),
so that the oracle and the CUDA path can both consume its output.

Every stream is keyed by (workload seed, round, request, stream id) through
numpy's SeedSequence, so any single request can be regenerated on its own —
the sampled-parity tests and the CPU baseline rely on that.

The workloads restate the five configurations this project is measured on;
their distributions follow the DSpark round as the pages describe it: base
logits U from the parallel backbone, bf16 Markov factors W1 [V, r] and
W2 [r, V] ("DSpark" page §2.3), hidden states h and the confidence weight w
(§3.1), an SPS(B) cost table (§4.1), and target logits built from U, the
Markov bias of the drafted prefix and Gaussian noise.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# stream ids (arbitrary, fixed)
_S_W1, _S_W2, _S_W = 11, 12, 13
_S_ANCHOR = 21
_S_U, _S_H, _S_TNOISE, _S_BONUS, _S_FAKE = 31, 32, 33, 34, 35
_S_WLM = 14


@dataclass(frozen=True)
class Workload:
    name: str
    R: int
    gamma: int
    V: int
    rank: int
    d: int
    seed: int
    u_std: float
    bump: str                   # "spikes": +6 on 2 ids per row; "zipf": 8 / i**1.1 on 64 ids
    w_std: float                # std of the bf16 W1 / W2 entries
    t_noise: tuple              # target-noise std for (first half, second half) of requests
    temperatures: tuple
    sps: str                    # "p2": page-2 cost model; "staircase": 3 cliffs
    modes: tuple = (0,)         # scheduler modes exercised: 0 early stop, 1 top-K, 2 fixed
    rounds: int = 1
    h_std: float = 1.0
    conf_w_std: float = 0.02

    @property
    def B_max(self) -> int:
        return self.R * (1 + self.gamma)


WORKLOADS = {
    "tiny_r4_g7_v4096": Workload("tiny_r4_g7_v4096", R=4, gamma=7, V=4096, rank=256, d=512, seed=0,
                                 u_std=2.0, bump="spikes", w_std=0.05, t_noise=(0.5, 0.5),
                                 temperatures=(1.0, 0.0), sps="p2", modes=(0,)),
    "r32_g7_v151936": Workload("r32_g7_v151936", R=32, gamma=7, V=151936, rank=256, d=2560,
                                seed=1, u_std=3.0, bump="zipf", w_std=0.03, t_noise=(1.0, 1.0),
                                temperatures=(1.0,), sps="p2", modes=(2,)),
    "r128_g16_v151936": Workload("r128_g16_v151936", R=128, gamma=16, V=151936, rank=256,
                                     d=4096, seed=2, u_std=3.0, bump="zipf", w_std=0.03,
                                     t_noise=(1.0, 1.0), temperatures=(1.0,), sps="p2",
                                     modes=(0,)),
    "r512_g16_v32768_staircase": Workload("r512_g16_v32768_staircase", R=512, gamma=16, V=32768,
                                       rank=256, d=2048, seed=3, u_std=3.0, bump="zipf",
                                       w_std=0.03, t_noise=(0.3, 2.0), temperatures=(1.0,),
                                       sps="staircase", modes=(0, 1), rounds=8),
    "r256_g16_v129280_d7168": Workload("r256_g16_v129280_d7168", R=256, gamma=16, V=129280,
                                       rank=256, d=7168, seed=4, u_std=3.0, bump="zipf",
                                       w_std=0.03, t_noise=(1.0, 1.0),
                                       temperatures=(0.0, 0.7, 1.0), sps="p2", modes=(0,)),
}
# the five workloads in the order the project lists them
ORDER = ["tiny_r4_g7_v4096", "r32_g7_v151936", "r128_g16_v151936",
         "r512_g16_v32768_staircase", "r256_g16_v129280_d7168"]


def scaled(base: Workload, **changes) -> Workload:
    """A copy of a workload with some sizes changed (parity cases)."""
    d = dict(base.__dict__)
    d.update(changes)
    if "name" not in changes:
        d["name"] = base.name + "_" + "_".join(f"{k}{v}" for k, v in changes.items())
    return Workload(**d)


def _rng(*key) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(k) for k in key]))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    # finite inputs only: the rounding increment cannot carry out of 32 bits
    b = np.ascontiguousarray(x, np.float32).view(np.uint32)
    b = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def weights(wl: Workload):
    """W1 bf16 [V, r], W2 bf16 [r, V], w fp32 [d + r]."""
    W1 = to_bf16_bits(_rng(wl.seed, _S_W1).standard_normal((wl.V, wl.rank), np.float32) * wl.w_std)
    W2 = to_bf16_bits(_rng(wl.seed, _S_W2).standard_normal((wl.rank, wl.V), np.float32) * wl.w_std)
    w = (_rng(wl.seed, _S_W).standard_normal(wl.d + wl.rank, np.float32) * wl.conf_w_std)
    return W1, W2, w.astype(np.float32)


def lm_head_weight(wl: Workload, rows_per_block: int = 256) -> np.ndarray:
    """W_lm bf16 bits [d, V] for the fused LM-head draft: normal entries scaled
    so that h . W_lm has the spread of the workload's base logits
    (u_std / (h_std * sqrt(d))).  Drawn in blocks of rows to bound the host
    memory at full size."""
    scale = np.float32(wl.u_std / (wl.h_std * np.sqrt(wl.d)))
    out = np.empty((wl.d, wl.V), np.uint16)
    for i0 in range(0, wl.d, rows_per_block):
        i1 = min(wl.d, i0 + rows_per_block)
        g = _rng(wl.seed, _S_WLM, i0)
        out[i0:i1] = to_bf16_bits(g.standard_normal((i1 - i0, wl.V), np.float32) * scale)
    return out


def anchors(wl: Workload, rnd: int = 0) -> np.ndarray:
    return _rng(wl.seed, _S_ANCHOR, rnd).integers(0, wl.V, wl.R, dtype=np.int64).astype(np.int32)


def _bump_rows(rng: np.random.Generator, rows: np.ndarray, wl: Workload) -> None:
    n, V = rows.shape
    if wl.bump == "spikes":
        for i in range(n):
            ids = rng.choice(V, 2, replace=False)
            rows[i, ids] += np.float32(6.0)
    elif wl.bump == "zipf":
        k = min(64, V)
        heights = (8.0 / np.arange(1, k + 1, dtype=np.float64) ** 1.1).astype(np.float32)
        for i in range(n):
            ids = rng.choice(V, k, replace=False)
            rows[i, ids] += heights
    else:
        raise ValueError(wl.bump)


def base_logits(wl: Workload, rnd: int, r: int, rows: int | None = None) -> np.ndarray:
    """U for request r: fp32 [gamma, V] (or `rows` rows)."""
    n = wl.gamma if rows is None else rows
    g = _rng(wl.seed, _S_U, rnd, r)
    U = g.standard_normal((n, wl.V), np.float32) * np.float32(wl.u_std)
    _bump_rows(g, U, wl)
    return U


def hidden(wl: Workload, rnd: int, r: int) -> np.ndarray:
    """h for request r: bf16 bits [gamma, d]."""
    g = _rng(wl.seed, _S_H, rnd, r)
    return to_bf16_bits(g.standard_normal((wl.gamma, wl.d), np.float32) * np.float32(wl.h_std))


def target_noise(wl: Workload, rnd: int, r: int) -> np.ndarray:
    """Target noise for request r: fp32 [gamma + 1, V]; std by request half."""
    std = wl.t_noise[0] if r < wl.R // 2 else wl.t_noise[1]
    g = _rng(wl.seed, _S_TNOISE, rnd, r)
    return g.standard_normal((wl.gamma + 1, wl.V), np.float32) * np.float32(std)


def bonus_base(wl: Workload, rnd: int, r: int) -> np.ndarray:
    """A fresh U-distributed row: the base of target row gamma (the bonus row)."""
    g = _rng(wl.seed, _S_BONUS, rnd, r)
    row = g.standard_normal((1, wl.V), np.float32) * np.float32(wl.u_std)
    _bump_rows(g, row, wl)
    return row[0]


def compose_target(U_r: np.ndarray, bias_r: np.ndarray, noise_r: np.ndarray,
                   bonus_r: np.ndarray) -> np.ndarray:
    """Target logits [gamma + 1, V] = U + bias of the drafted prefix + noise,
    and row gamma = a fresh U-distributed row + noise.  bias_r [gamma, V] is
    computed by the caller."""
    g, V = U_r.shape
    T = np.empty((g + 1, V), np.float32)
    T[:g] = (U_r.astype(np.float64) + bias_r + noise_r[:g]).astype(np.float32)
    T[g] = (bonus_r.astype(np.float64) + noise_r[g]).astype(np.float32)
    return T


def fake_draft(wl: Workload, rnd: int, r: int):
    """Stand-in draft outputs (tokens, p_d(x), log Z) for requests a test does
    not compare: they only have to be valid inputs."""
    g = _rng(wl.seed, _S_FAKE, rnd, r)
    tokens = g.integers(0, wl.V, wl.gamma, dtype=np.int64).astype(np.int32)
    pd = g.uniform(0.05, 1.0, wl.gamma).astype(np.float32)
    logZ = g.uniform(10.0, 20.0, wl.gamma).astype(np.float32)
    return tokens, pd, logZ


def sps_table(wl: Workload) -> np.ndarray:
    """SPS(B) for B = 0 .. R (1 + gamma), fp64, indexed by B.

    "p2": 1 / max(16e9 / (3.35e12 * 0.8), B * 16e9 / (989e12 * 0.5)), the
    page-2 H100 cost model of an 8B model (verify forward only).
    "staircase": 1000 steps/s, slowed by 25 % / 50 % / 100 % of the base step
    time once B reaches 1024 / 2048 / 4096 — three cliffs, so Theta is not
    unimodal in the budget."""
    B = np.arange(wl.B_max + 1, dtype=np.float64)
    if wl.sps == "p2":
        mem = 16e9 / (3.35e12 * 0.8)
        comp = B * 16e9 / (989e12 * 0.5)
        return 1.0 / np.maximum(mem, comp)
    if wl.sps == "staircase":
        slow = 1.0 + 0.25 * (B >= 1024) + 0.5 * (B >= 2048) + 1.0 * (B >= 4096)
        return 1000.0 / slow
    raise ValueError(wl.sps)


@dataclass
class RoundInputs:
    """Host arrays for one round of a workload (requests in `requests`)."""
    U: np.ndarray            # fp32 [n, gamma, V]
    h: np.ndarray            # bf16 bits [n, gamma, d]
    anchors: np.ndarray      # int32 [n]
    requests: np.ndarray     # int64 [n]
    extras: dict = field(default_factory=dict)


def round_inputs(wl: Workload, rnd: int = 0, requests=None, anchor_override=None) -> RoundInputs:
    req = np.arange(wl.R) if requests is None else np.asarray(requests, np.int64)
    U = np.empty((len(req), wl.gamma, wl.V), np.float32)
    h = np.empty((len(req), wl.gamma, wl.d), np.uint16)
    for i, r in enumerate(req):
        U[i] = base_logits(wl, rnd, int(r))
        h[i] = hidden(wl, rnd, int(r))
    anc_all = anchors(wl, rnd) if anchor_override is None else np.asarray(anchor_override, np.int32)
    return RoundInputs(U=U, h=h, anchors=anc_all[req].astype(np.int32), requests=req)
