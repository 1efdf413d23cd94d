"""Analytical cost model of the "投机解码的新做法" page, section "负载越高，K 越要小"
(test infrastructure; restated from what the page computes, not from its listing).

An 8B-parameter bf16 model on an H100: every forward step reads all weights
once (16 GB at 80 % of 3.35 TB/s) or, when the step holds many tokens, is
bound by 2 * 8e9 FLOPs per token at 50 % of 989 TFLOP/s.  A draft forward
costs 0.25 ms; each further draft position is accepted with probability 0.8
given that all earlier ones were.

The page derives from this model both its best-K table and the SPS(B) curve
its adaptive-verification planner optimises; configs 0, 2 and 4 of this
project use the same SPS(B) = 1 / max(W/BW, B F / FLOPS) table.
"""
from __future__ import annotations

WEIGHT_BYTES = 16e9
EFFECTIVE_BW = 3.35e12 * 0.8
FLOPS_PER_TOKEN = 2 * 8e9
EFFECTIVE_FLOPS = 989e12 * 0.5
DRAFT_SECONDS = 0.25e-3
ACCEPT_PROB = 0.8


def step_seconds(tokens: float) -> float:
    """Time of one target forward over `tokens` tokens: the larger of the
    weight-streaming time and the arithmetic time."""
    memory_time = WEIGHT_BYTES / EFFECTIVE_BW
    compute_time = tokens * FLOPS_PER_TOKEN / EFFECTIVE_FLOPS
    return memory_time if memory_time >= compute_time else compute_time


def expected_accepted(k: int, alpha: float = ACCEPT_PROB) -> float:
    """Expected accepted draft tokens with k drafted positions: the j-th is
    kept with probability alpha**j (all earlier ones must be kept)."""
    total = 0.0
    survive = 1.0
    for _ in range(k):
        survive *= alpha
        total += survive
    return total


def tokens_per_second(batch: int, k: int, one_shot_draft: bool) -> float:
    """Output tokens per second of `batch` requests each drafting k tokens:
    a draft phase (k sequential draft forwards, or one block forward) plus
    one verify forward over batch * (1 + k) tokens; each request yields the
    accepted drafts plus the one token the verify step always adds."""
    if k == 0:
        draft_time = 0.0
    elif one_shot_draft:
        draft_time = DRAFT_SECONDS
    else:
        draft_time = k * DRAFT_SECONDS
    produced = batch * (1.0 + expected_accepted(k))
    return produced / (draft_time + step_seconds(batch * (1 + k)))


def best_k(batch: int, one_shot_draft: bool, k_max: int = 8) -> int:
    """Smallest k in [0, k_max] with the highest throughput."""
    best = 0
    best_rate = tokens_per_second(batch, 0, one_shot_draft)
    for k in range(1, k_max + 1):
        rate = tokens_per_second(batch, k, one_shot_draft)
        if rate > best_rate:
            best, best_rate = k, rate
    return best


def sps_target_only(tokens: float) -> float:
    """Steps per second of the verify forward alone (configs 0, 2, 4)."""
    return 1.0 / step_seconds(tokens)


def sps_with_draft(tokens: float) -> float:
    """Steps per second of one draft forward plus the verify forward: the
    rate the page's adaptive-verification planner divides by."""
    return 1.0 / (DRAFT_SECONDS + step_seconds(tokens))
