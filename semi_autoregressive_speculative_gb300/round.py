"""One DSpark round on device memory: buffers plus the four calls.

``DeviceRound`` owns the device tensors of one workload shape (inputs,
outputs, scratch workspace) and runs the round through the C ABI on the
current torch stream: draft -> confidence -> schedule -> verify.  Target
logits are an input of verify and are set by the caller, on the device or,
for the admitted rows only, from page-locked host memory (load_target_rows).
"""
from __future__ import annotations

import numpy as np
import torch

from . import (MODE_EARLY_STOP, MODE_FIXED, MODE_TOP_K, dspark_clear_status, dspark_confidence,
               dspark_load_verified_rows, dspark_markov_draft, dspark_schedule, dspark_verify, dspark_workspace_size,
               read_status)

__all__ = ["DeviceRound", "MODE_EARLY_STOP", "MODE_TOP_K", "MODE_FIXED"]


def _host(x, as_int16: bool = False) -> torch.Tensor:
    a = np.ascontiguousarray(x)
    if as_int16:
        a = a.view(np.int16)  # bf16 bit patterns travel as int16
    return torch.from_numpy(a)


class DeviceRound:
    def __init__(self, R: int, gamma: int, V: int, rank: int, d: int, device="cuda:0"):
        self.R, self.gamma, self.V, self.rank, self.d = R, gamma, V, rank, d
        self.device = torch.device(device)
        dv = self.device
        f32, i32 = torch.float32, torch.int32
        self.U = torch.empty((R, gamma, V), dtype=f32, device=dv)
        self.T = torch.empty((R, gamma + 1, V), dtype=f32, device=dv)
        self.h = torch.empty((R, gamma, d), dtype=torch.int16, device=dv)
        self.W1 = torch.empty((V, rank), dtype=torch.int16, device=dv)
        self.W2 = torch.empty((rank, V), dtype=torch.int16, device=dv)
        self.w = torch.empty((d + rank,), dtype=f32, device=dv)
        self.anchors = torch.empty((R,), dtype=i32, device=dv)
        self.sps = torch.empty((R * (1 + gamma) + 1,), dtype=torch.float64, device=dv)
        self.tokens = torch.empty((R, gamma), dtype=i32, device=dv)
        self.pd = torch.empty((R, gamma), dtype=f32, device=dv)
        self.logZ = torch.empty((R, gamma), dtype=f32, device=dv)
        self.c = torch.empty((R, gamma), dtype=f32, device=dv)
        self.a = torch.empty((R, gamma), dtype=f32, device=dv)
        self.lens = torch.empty((R,), dtype=i32, device=dv)
        self.sched_out = torch.zeros((2,), dtype=i32, device=dv)   # total_b, argmax_b
        self.theta = torch.zeros((1,), dtype=torch.float64, device=dv)
        self.n_accept = torch.empty((R,), dtype=i32, device=dv)
        self.next_token = torch.empty((R,), dtype=i32, device=dv)
        self.c_star = torch.empty((R, gamma), dtype=f32, device=dv)
        ws = dspark_workspace_size(R, gamma, V, rank, d)
        if ws == 0:
            raise ValueError("invalid sizes")
        self.workspace = torch.zeros((ws,), dtype=torch.uint8, device=dv)

    # ------------------------------------------------------------ inputs
    def set_weights(self, W1, W2, w):
        self.W1.copy_(_host(W1, True))
        self.W2.copy_(_host(W2, True))
        self.w.copy_(_host(np.asarray(w, np.float32)))

    def set_round(self, U, h, anchors, sps=None):
        self.U.copy_(_host(np.asarray(U, np.float32)))
        self.h.copy_(_host(h, True))
        self.anchors.copy_(_host(np.asarray(anchors, np.int32)))
        if sps is not None:
            self.sps.copy_(_host(np.asarray(sps, np.float64)))

    # ------------------------------------------------------------ the four steps
    def draft(self, temperature: float, seed: int, rnd: int):
        dspark_markov_draft(self.U, self.W1, self.W2, self.anchors, temperature, seed, rnd, self.tokens, self.pd,
                            self.logZ, self.workspace)

    def confidence(self, tokens=None, sts_temperature=None):
        dspark_confidence(self.h, self.W1, self.w, self.anchors, self.tokens if tokens is None else tokens,
                          self.c, self.a, self.workspace, sts_temperature=sts_temperature)

    def schedule(self, mode: int, budget_K: int = 0, a=None):
        dspark_schedule(self.a if a is None else a, self.sps, mode, budget_K, self.lens, self.sched_out[0:1],
                        self.sched_out[1:2], self.theta, self.workspace)

    def load_target_rows(self, T_host):
        """Copy rows 0..lens[r] of each request from the page-locked host
        tensor T_host [R, gamma+1, V] into self.T (lens stays on the device)."""
        dspark_load_verified_rows(T_host, self.lens, self.T, self.workspace)

    def verify(self, temperature: float, seed: int, rnd: int, tokens=None, pd=None, logZ=None, lens=None,
               c_star: bool = False):
        """c_star=True also writes the analytic acceptance into self.c_star."""
        dspark_verify(self.T, self.U, self.W1, self.W2, self.anchors, self.tokens if tokens is None else tokens,
                      self.pd if pd is None else pd, self.logZ if logZ is None else logZ,
                      self.lens if lens is None else lens, temperature, seed, rnd, self.n_accept,
                      self.next_token, self.workspace, c_star=self.c_star if c_star else None)

    def clear_status(self):
        dspark_clear_status(self.workspace)

    def status(self) -> int:
        return read_status(self.workspace)
