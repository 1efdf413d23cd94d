"""Python binding of libdspark.so: the DSpark speculative-decoding round on
one GB300.

Argument marshalling only — every step of the round runs in the library's
CUDA kernels.  Functions carry the C names of ``include/dspark.h`` and take
torch CUDA tensors (device memory) plus the current torch stream.  Loading
fails loudly when the library is missing: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libdspark.so")

DSPARK_OK = 0
DSPARK_ERR_INVALID_ARG = -1
DSPARK_ERR_UNSUPPORTED_SHAPE = -2
DSPARK_ERR_CUDA = -3
DSPARK_ERR_STATIC_SCRATCH_TOO_SMALL = -4
DSPARK_NOALLOC_SCRATCH_BYTES = 16 << 20
DSPARK_STATUS_NONFINITE = 1
DSPARK_STATUS_BAD_TOKEN = 2
DSPARK_STATUS_TIMEOUT = 4
DSPARK_STATUS_BAD_LENGTH = 8
MODE_EARLY_STOP, MODE_TOP_K, MODE_FIXED = 0, 1, 2

EXPORTS = ("dspark_workspace_size", "dspark_clear_status", "dspark_markov_draft", "dspark_confidence",
           "dspark_schedule", "dspark_verify", "dspark_markov_draft_noalloc", "dspark_selftest_bounded_wait",
           "dspark_markov_draft_lmhead", "dspark_load_verified_rows")

_lib = None


class DsparkError(RuntimeError):
    def __init__(self, fn: str, code: int):
        names = {-1: "DSPARK_ERR_INVALID_ARG", -2: "DSPARK_ERR_UNSUPPORTED_SHAPE", -3: "DSPARK_ERR_CUDA",
                 -4: "DSPARK_ERR_STATIC_SCRATCH_TOO_SMALL"}
        super().__init__(f"{fn} returned {names.get(code, code)}")
        self.code = code


def lib() -> ctypes.CDLL:
    """Load libdspark.so (build it first with ``build.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libdspark.so not built at {LIB_PATH}; run "
                              "python -m semi_autoregressive_speculative_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        U64, U32, SZ = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_size_t
        L.dspark_workspace_size.restype = SZ
        L.dspark_workspace_size.argtypes = [I, I, I, I, I]
        L.dspark_clear_status.restype = I
        L.dspark_clear_status.argtypes = [P, P]
        L.dspark_selftest_bounded_wait.restype = I
        L.dspark_selftest_bounded_wait.argtypes = [P, P]
        L.dspark_markov_draft.restype = I
        L.dspark_markov_draft.argtypes = [P, P, P, P, I, I, I, I, F, U64, U32, P, P, P, P, SZ, P]
        L.dspark_markov_draft_lmhead.restype = I
        L.dspark_markov_draft_lmhead.argtypes = [P, P, P, P, P, I, I, I, I, I, F, U64, U32, P, P, P, P, SZ, P]
        L.dspark_confidence.restype = I
        L.dspark_confidence.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, P, SZ, P]
        L.dspark_schedule.restype = I
        L.dspark_schedule.argtypes = [P, I, I, P, I, I, I, P, P, P, P, P, SZ, P]
        L.dspark_verify.restype = I
        L.dspark_verify.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, F, U64, U32, P, P, P, P, SZ, P]
        L.dspark_load_verified_rows.restype = I
        L.dspark_load_verified_rows.argtypes = [P, P, I, I, I, P, P, P]
        L.dspark_markov_draft_noalloc.restype = I
        L.dspark_markov_draft_noalloc.argtypes = [P, P, P, P, I, I, I, I, F, U64, U32, P, P, P, P, P]
        _lib = L
    return _lib


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _check(fn: str, rc: int) -> None:
    if rc != DSPARK_OK:
        raise DsparkError(fn, rc)


def dspark_workspace_size(R: int, gamma: int, V: int, rank: int, d: int) -> int:
    return lib().dspark_workspace_size(R, gamma, V, rank, d)


def dspark_clear_status(workspace, stream=None) -> None:
    _check("dspark_clear_status", lib().dspark_clear_status(_ptr(workspace), _stream(stream)))


def dspark_selftest_bounded_wait(workspace, stream=None) -> None:
    """Enqueue the timeout self-test: a bounded device wait that gives up and
    sets DSPARK_STATUS_TIMEOUT in the workspace status word (about 2 s)."""
    _check("dspark_selftest_bounded_wait", lib().dspark_selftest_bounded_wait(_ptr(workspace), _stream(stream)))


def read_status(workspace) -> int:
    """Device status word (first int32 of the workspace); synchronises."""
    return int(workspace[:4].view(dtype=__import__("torch").int32).item())


def dspark_markov_draft(U, W1, W2, anchors, temperature, seed, round_, tokens, pd_tok, logZ, workspace,
                        stream=None) -> None:
    R, gamma, V = U.shape
    rank = W1.shape[1]
    _check("dspark_markov_draft", lib().dspark_markov_draft(
        _ptr(U), _ptr(W1), _ptr(W2), _ptr(anchors), R, gamma, V, rank, float(temperature), int(seed),
        int(round_), _ptr(tokens), _ptr(pd_tok), _ptr(logZ), _ptr(workspace), _nbytes(workspace),
        _stream(stream)))


def dspark_markov_draft_lmhead(h, W_lm, W1, W2, anchors, temperature, seed, round_, tokens, pd_tok, logZ, workspace,
                               stream=None) -> None:
    """The draft with the LM head fused in: h [R, gamma, d] bf16 and W_lm
    [d, V] bf16 in place of U (see include/dspark.h)."""
    R, gamma, d = h.shape
    V = W_lm.shape[1]
    rank = W1.shape[1]
    _check("dspark_markov_draft_lmhead", lib().dspark_markov_draft_lmhead(
        _ptr(h), _ptr(W_lm), _ptr(W1), _ptr(W2), _ptr(anchors), R, gamma, V, rank, d, float(temperature), int(seed),
        int(round_), _ptr(tokens), _ptr(pd_tok), _ptr(logZ), _ptr(workspace), _nbytes(workspace), _stream(stream)))


def dspark_confidence(h, W1, w, anchors, tokens, c, a, workspace, stream=None, sts_temperature=None) -> None:
    R, gamma, d = h.shape
    V, rank = W1.shape
    if sts_temperature is not None and tuple(sts_temperature.shape) != (gamma,):
        raise ValueError(f"sts_temperature must have shape ({gamma},), got {tuple(sts_temperature.shape)}")
    _check("dspark_confidence", lib().dspark_confidence(
        _ptr(h), _ptr(W1), _ptr(w), _ptr(sts_temperature), _ptr(anchors), _ptr(tokens), R, gamma, d, rank, V, _ptr(c), _ptr(a),
        _ptr(workspace), _nbytes(workspace), _stream(stream)))


def dspark_schedule(a, sps, mode, budget_K, lens, total_b, argmax_b, theta, workspace, stream=None) -> None:
    R, gamma = a.shape
    _check("dspark_schedule", lib().dspark_schedule(
        _ptr(a), R, gamma, _ptr(sps), sps.shape[0], int(mode), int(budget_K), _ptr(lens), _ptr(total_b),
        _ptr(argmax_b), _ptr(theta), _ptr(workspace), _nbytes(workspace), _stream(stream)))


def dspark_verify(T, U, W1, W2, anchors, tokens, pd_tok, logZ, lens, temperature, seed, round_, n_accept,
                  next_token, workspace, stream=None, c_star=None) -> None:
    """`c_star`: optional fp32 [R, gamma] device tensor for the analytic acceptance."""
    R, gamma, V = U.shape
    rank = W1.shape[1]
    if c_star is not None and tuple(c_star.shape) != (R, gamma):
        raise ValueError(f"c_star must have shape ({R}, {gamma}), got {tuple(c_star.shape)}")
    _check("dspark_verify", lib().dspark_verify(
        _ptr(T), _ptr(U), _ptr(W1), _ptr(W2), _ptr(anchors), _ptr(tokens), _ptr(pd_tok), _ptr(logZ),
        _ptr(lens), R, gamma, V, rank, float(temperature), int(seed), int(round_), _ptr(n_accept),
        _ptr(next_token), _ptr(c_star), _ptr(workspace), _nbytes(workspace), _stream(stream)))


def dspark_load_verified_rows(T_host, lens, T, workspace, stream=None) -> None:
    """`T_host`: page-locked CPU fp32 tensor [R, gamma+1, V]; `lens`, `T` and
    `workspace` on the device."""
    R, g1, V = T.shape
    if tuple(T_host.shape) != (R, g1, V):
        raise ValueError(f"T_host must have shape {(R, g1, V)}, got {tuple(T_host.shape)}")
    _check("dspark_load_verified_rows", lib().dspark_load_verified_rows(
        _ptr(T_host), _ptr(lens), R, g1 - 1, V, _ptr(T), _ptr(workspace), _stream(stream)))


def dspark_markov_draft_noalloc(U, W1, W2, anchors, temperature, seed, round_, tokens, pd_tok, logZ, status=None,
                                stream=None) -> None:
    """The draft without a workspace: scratch lives in the library's own
    16 MiB device array (see include/dspark.h).  `status`, if given, is a
    device int32 tensor that receives this call's status bits."""
    R, gamma, V = U.shape
    rank = W1.shape[1]
    _check("dspark_markov_draft_noalloc", lib().dspark_markov_draft_noalloc(
        _ptr(U), _ptr(W1), _ptr(W2), _ptr(anchors), R, gamma, V, rank, float(temperature), int(seed),
        int(round_), _ptr(tokens), _ptr(pd_tok), _ptr(logZ), _ptr(status), _stream(stream)))
