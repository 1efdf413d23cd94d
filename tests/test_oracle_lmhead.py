"""Pins of the oracle's LM head, U = h . W_lm (the fused LM-head draft's
logits: "DSpark: Speculative decodingを活用した…", "実サービス配備 › 拡張可能な学習
› 隠れ状態通信").  Each pin is fixed by the mathematics, not by the oracle's
own arithmetic: a one-hot W_lm is a column gather of h, integer-valued inputs
give the exact integer product, and a sum that fp32 accumulation rounds twice
is rounded once."""
import numpy as np

import oracle as orc


def _bits(x):
    """bf16 bit patterns of values that bf16 holds exactly (test inputs only)."""
    b = np.asarray(x, np.float32).view(np.uint32)
    assert np.all((b & 0xFFFF) == 0)
    return (b >> 16).astype(np.uint16)


def test_one_hot_columns_gather_h():
    rng = np.random.default_rng(5)
    d, V = 40, 97
    h = rng.standard_normal((3, 4, d)).astype(np.float32)
    h = ((h.view(np.uint32) & 0xFFFF0000).view(np.float32))  # bf16-exact values
    perm = rng.integers(0, d, V)
    W = np.zeros((d, V), np.float32)
    W[perm, np.arange(V)] = 1.0
    U = orc.lm_head_logits(_bits(h), _bits(W), cols_per_block=32)
    assert U.shape == (3, 4, V) and U.dtype == np.float32
    np.testing.assert_array_equal(U, h[..., perm])


def test_integer_inputs_give_the_exact_product():
    rng = np.random.default_rng(6)
    d, V = 300, 1000  # several column blocks and a ragged last one
    h = rng.integers(-8, 9, (2, 3, d))
    W = rng.integers(-8, 9, (d, V))
    U = orc.lm_head_logits(_bits(h), _bits(W), cols_per_block=256)
    exact = np.einsum("abk,kv->abv", h.astype(np.int64), W.astype(np.int64))
    np.testing.assert_array_equal(U, exact.astype(np.float32))


def test_each_sum_is_rounded_once():
    # 1 + 2^-24 + 2^-40 lies above the midpoint between 1 and 1 + 2^-23: one
    # rounding gives 1 + 2^-23, while summing in fp32 would give 1 (the first
    # addition ties to even)
    h = np.array([[1.0, 2.0 ** -24, 2.0 ** -40]], np.float32)
    W = np.ones((3, 2), np.float32)
    W[:, 1] = [1.0, -1.0, 0.0]
    U = orc.lm_head_logits(_bits(h), _bits(W))
    assert U[0, 0] == np.float32(1.0 + 2.0 ** -23)
    assert U[0, 1] == np.float32(1.0 - 2.0 ** -24)
