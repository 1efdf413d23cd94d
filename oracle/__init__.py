"""CPU oracle for one DSpark speculative-decoding round (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
product path never imports, links or executes anything here, and this package
never imports the product path.

The arithmetic lives in ``oracle.c`` (plain single-threaded C, fp64); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
The page-2 cost model and planner are restated in ``cost_model.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

# -ffp-contract=off: no fused multiply-add contraction, so x86 and aarch64
# hosts round every operation the same way.
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, no GPU needed)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int
        U64 = ctypes.c_uint64
        F = ctypes.c_float
        D = ctypes.c_double
        I32 = ctypes.c_int32
        sig = {
            "oracle_philox4x64_10": (None, [P, P, P]),
            "oracle_uniform": (D, [U64, U64, U64, U64, U64]),
            "oracle_markov_bias": (None, [P, P, I, I, I32, P]),
            "oracle_inverse_cdf": (I32, [P, I, D]),
            "oracle_draft_probs": (D, [P, P, P, I32, I, I, F, P]),
            "oracle_draft_logits_f32": (None, [P, P, P, I32, I, I, P]),
            "oracle_target_probs": (D, [P, I, F, P]),
            "oracle_draft_request": (I, [P, P, P, I32, I, I, I, F, U64, U64, U64, P, P, P]),
            "oracle_confidence_request": (I, [P, P, P, I32, P, I, I, I, I, P, P, P]),
            "oracle_survival": (None, [P, I, P]),
            "oracle_schedule": (I, [P, I, I, P, I, I, I, P, P, P, P, P]),
            "oracle_verify_request_u": (I, [P, P, P, P, I32, P, I, I, I, I, F, P, P, P, P]),
            "oracle_verify_request": (I, [P, P, P, P, I32, P, I, I, I, I, F, U64, U64, U64, P, P]),
            "oracle_verify_position": (I, [P, P, I, I32, D, D, P, P]),
            "oracle_overlap": (D, [P, P, I]),
            "oracle_c_star_request": (I, [P, P, P, P, I32, P, I, I, I, I, F, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


# ---------------------------------------------------------------- uniforms
def philox4x64_10(ctr, key) -> np.ndarray:
    c = _c(ctr, np.uint64)
    k = _c(key, np.uint64)
    out = np.zeros(4, np.uint64)
    lib().oracle_philox4x64_10(_p(c), _p(k), _p(out))
    return out


def uniform(seed: int, rnd: int, request: int, position: int, purpose: int) -> float:
    return lib().oracle_uniform(seed, rnd, request, position, purpose)


# ---------------------------------------------------------------- draft
def _bf16_f64(bits) -> np.ndarray:
    """bf16 bit patterns -> their exact values as fp64."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def lm_head_logits(h, W_lm, cols_per_block: int = 16384) -> np.ndarray:
    """U = h . W_lm, the logits the fused LM-head draft forms from the shipped
    pre-LM-head hidden state ("DSpark: Speculative decodingを活用した…",
    "実サービス配備 › 拡張可能な学習 › 隠れ状態通信": the hidden state, not the
    V-wide logits, crosses the wire and the LM head runs where the tokens are
    drawn).  The bf16 values are multiplied and summed in fp64 (numpy's
    matmul) and each sum is rounded once to fp32.  h bf16 bits [..., d], W_lm
    bf16 bits [d, V] -> fp32 [..., V]; W_lm is decoded in blocks of columns to
    bound the host memory."""
    hf = _bf16_f64(h)
    W_lm = np.asarray(W_lm, np.uint16)
    d, V = W_lm.shape
    assert hf.shape[-1] == d
    out = np.empty(hf.shape[:-1] + (V,), np.float32)
    for v0 in range(0, V, cols_per_block):
        v1 = min(V, v0 + cols_per_block)
        out[..., v0:v1] = (hf @ _bf16_f64(W_lm[:, v0:v1])).astype(np.float32)
    return out


def markov_bias(W1: np.ndarray, W2: np.ndarray, prev: int) -> np.ndarray:
    W1 = _c(W1, np.uint16)
    W2 = _c(W2, np.uint16)
    V, rank = W1.shape
    out = np.zeros(V, np.float64)
    lib().oracle_markov_bias(_p(W1), _p(W2), V, rank, int(prev), _p(out))
    return out


def draft_probs(U_row, W1, W2, prev: int, temperature: float):
    U_row = _c(U_row, np.float32)
    W1 = _c(W1, np.uint16)
    W2 = _c(W2, np.uint16)
    V, rank = W1.shape
    p = np.zeros(V, np.float64)
    logZ = lib().oracle_draft_probs(_p(U_row), _p(W1), _p(W2), int(prev), V, rank,
                                    float(temperature), _p(p))
    return p, logZ


def draft_logits_f32(U_row, W1, W2, prev: int) -> np.ndarray:
    U_row = _c(U_row, np.float32)
    W1 = _c(W1, np.uint16)
    W2 = _c(W2, np.uint16)
    V, rank = W1.shape
    z = np.zeros(V, np.float32)
    lib().oracle_draft_logits_f32(_p(U_row), _p(W1), _p(W2), int(prev), V, rank, _p(z))
    return z


def target_probs(T_row, temperature: float):
    T_row = _c(T_row, np.float32)
    p = np.zeros(T_row.shape[0], np.float64)
    logZ = lib().oracle_target_probs(_p(T_row), T_row.shape[0], float(temperature), _p(p))
    return p, logZ


def inverse_cdf(p, u: float) -> int:
    p = _c(p, np.float64)
    return lib().oracle_inverse_cdf(_p(p), p.shape[0], float(u))


def draft(U, W1, W2, anchors, temperature: float, seed: int, rnd: int, request_ids=None):
    """Draft every request of U [n, gamma, V]; request_ids[i] is the request
    index used in the Philox counter for row i (default: 0..n-1)."""
    U = _c(U, np.float32)
    W1 = _c(W1, np.uint16)
    W2 = _c(W2, np.uint16)
    n, gamma, V = U.shape
    rank = W1.shape[1]
    anchors = np.asarray(anchors, np.int32)
    ids = np.arange(n) if request_ids is None else np.asarray(request_ids)
    tokens = np.zeros((n, gamma), np.int32)
    pd = np.zeros((n, gamma), np.float32)
    logZ = np.zeros((n, gamma), np.float32)
    for i in range(n):
        t = np.zeros(gamma, np.int32)
        q = np.zeros(gamma, np.float32)
        z = np.zeros(gamma, np.float32)
        rc = lib().oracle_draft_request(_p(U[i]), _p(W1), _p(W2), int(anchors[i]), gamma, V, rank,
                                        float(temperature), seed, rnd, int(ids[i]), _p(t), _p(q),
                                        _p(z))
        _check(rc, "draft")
        tokens[i], pd[i], logZ[i] = t, q, z
    return tokens, pd, logZ


# ---------------------------------------------------------------- confidence
def confidence(h, W1, w, anchors, tokens, sts_temperature=None):
    """c, a of every request; sts_temperature: per-position temperatures
    [gamma] that divide the confidence logits (None: no scaling)."""
    sts = None if sts_temperature is None else _c(sts_temperature, np.float32)
    h = _c(h, np.uint16)
    W1 = _c(W1, np.uint16)
    w = _c(w, np.float32)
    tokens = _c(tokens, np.int32)
    n, gamma, d = h.shape
    V, rank = W1.shape
    c = np.zeros((n, gamma), np.float32)
    a = np.zeros((n, gamma), np.float32)
    for i in range(n):
        ci = np.zeros(gamma, np.float32)
        ai = np.zeros(gamma, np.float32)
        rc = lib().oracle_confidence_request(_p(h[i]), _p(W1), _p(w), int(anchors[i]),
                                             _p(tokens[i]), gamma, d, rank, V,
                                             None if sts is None else _p(sts), _p(ci), _p(ai))
        _check(rc, "confidence")
        c[i], a[i] = ci, ai
    return c, a


def survival(c) -> np.ndarray:
    """a = running fp32 product of c along the last axis."""
    c = _c(c, np.float32)
    flat = c.reshape(-1, c.shape[-1])
    a = np.zeros_like(flat)
    for i in range(flat.shape[0]):
        lib().oracle_survival(_p(flat[i]), flat.shape[1], _p(a[i]))
    return a.reshape(c.shape)


# ---------------------------------------------------------------- scheduler
MODE_EARLY_STOP, MODE_TOP_K, MODE_FIXED = 0, 1, 2


def schedule(a, sps, mode: int, budget_K: int = 0):
    a = _c(a, np.float32)
    sps = _c(sps, np.float64)
    R, gamma = a.shape
    lens = np.zeros(R, np.int32)
    total_b = ctypes.c_int32()
    argmax_b = ctypes.c_int32()
    theta = ctypes.c_double()
    theta_all = np.zeros(R * gamma + 1, np.float64)
    rc = lib().oracle_schedule(_p(a), R, gamma, _p(sps), sps.shape[0], int(mode), int(budget_K),
                               _p(lens), ctypes.addressof(total_b), ctypes.addressof(argmax_b),
                               ctypes.addressof(theta), _p(theta_all))
    _check(rc, "schedule")
    return dict(lens=lens, total_b=total_b.value, argmax_b=argmax_b.value, theta=theta.value,
                theta_all=theta_all)


# ---------------------------------------------------------------- verify
def verify(T, U, W1, W2, anchors, tokens, lens, temperature: float, seed: int, rnd: int,
           request_ids=None):
    """T [n, gamma+1, V], U [n, gamma, V]; returns (n_accept, next_token)."""
    T = _c(T, np.float32)
    U = _c(U, np.float32)
    W1 = _c(W1, np.uint16)
    W2 = _c(W2, np.uint16)
    tokens = _c(tokens, np.int32)
    n, gamma, V = U.shape
    rank = W1.shape[1]
    ids = np.arange(n) if request_ids is None else np.asarray(request_ids)
    n_acc = np.zeros(n, np.int32)
    nxt = np.zeros(n, np.int32)
    for i in range(n):
        a = ctypes.c_int32()
        t = ctypes.c_int32()
        rc = lib().oracle_verify_request(_p(T[i]), _p(U[i]), _p(W1), _p(W2), int(anchors[i]),
                                         _p(tokens[i]), int(lens[i]), gamma, V, rank,
                                         float(temperature), seed, rnd, int(ids[i]),
                                         ctypes.addressof(a), ctypes.addressof(t))
        _check(rc, "verify")
        n_acc[i], nxt[i] = a.value, t.value
    return n_acc, nxt


def verify_request_u(T_r, U_r, W1, W2, anchor: int, tokens_r, length: int, temperature: float,
                     u_acc, u_res):
    T_r = _c(T_r, np.float32)
    U_r = _c(U_r, np.float32)
    W1 = _c(W1, np.uint16)
    W2 = _c(W2, np.uint16)
    tokens_r = _c(tokens_r, np.int32)
    u_acc = _c(u_acc, np.float64)
    u_res = _c(u_res, np.float64)
    gamma, V = U_r.shape
    a = ctypes.c_int32()
    t = ctypes.c_int32()
    rc = lib().oracle_verify_request_u(_p(T_r), _p(U_r), _p(W1), _p(W2), int(anchor), _p(tokens_r),
                                       int(length), gamma, V, W1.shape[1], float(temperature),
                                       _p(u_acc), _p(u_res), ctypes.addressof(a),
                                       ctypes.addressof(t))
    _check(rc, "verify_request_u")
    return a.value, t.value


def verify_position(pt, pd, x: int, u_acc: float, u_res: float):
    pt = _c(pt, np.float64)
    pd = _c(pd, np.float64)
    acc = ctypes.c_int32()
    tok = ctypes.c_int32()
    rc = lib().oracle_verify_position(_p(pt), _p(pd), pt.shape[0], int(x), float(u_acc),
                                      float(u_res), ctypes.addressof(acc), ctypes.addressof(tok))
    _check(rc, "verify_position")
    return acc.value, tok.value


def overlap(pd, pt) -> float:
    pd = _c(pd, np.float64)
    pt = _c(pt, np.float64)
    return lib().oracle_overlap(_p(pd), _p(pt), pd.shape[0])


def c_star(T, U, W1, W2, anchors, tokens, lens, temperature: float) -> np.ndarray:
    """Analytic acceptance c* [n, gamma] (fp64) of every position j <= lens[i]
    with j < gamma; NaN elsewhere."""
    T = _c(T, np.float32)
    U = _c(U, np.float32)
    W1 = _c(W1, np.uint16)
    W2 = _c(W2, np.uint16)
    tokens = _c(tokens, np.int32)
    n, gamma, V = U.shape
    out = np.empty((n, gamma), np.float64)
    for i in range(n):
        row = np.empty(gamma, np.float64)
        rc = lib().oracle_c_star_request(_p(T[i]), _p(U[i]), _p(W1), _p(W2), int(anchors[i]),
                                         _p(tokens[i]), int(lens[i]), gamma, V, W1.shape[1],
                                         float(temperature), _p(row))
        _check(rc, "c_star")
        out[i] = row
    return out
