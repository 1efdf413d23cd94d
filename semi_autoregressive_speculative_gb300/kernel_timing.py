"""Back-to-back timing of single library calls (a profiling tool).

    python -m semi_autoregressive_speculative_gb300.kernel_timing confidence [--calls 40]
    python -m semi_autoregressive_speculative_gb300.kernel_timing verify [--calls 20]
    python -m semi_autoregressive_speculative_gb300.kernel_timing lmhead [--calls 5]

``confidence``: dspark_confidence at the batch-128 shape (R=128, gamma=16,
d=4096) and at R=256, gamma=16, d=7168, called back to back on rotating h
buffers whose total exceeds the L2, so that h streams from HBM as it does in a
round; CUDA events around the whole run.  ``verify``: dspark_verify, plain and
with the optional c* output, on the batch-128 workload's own state (draft,
synthetic target logits, confidence and early-stop schedule), CUDA events
around each call.  ``lmhead``: dspark_markov_draft_lmhead at the batch-128
shape (R=128, gamma=16, V=151936, d=4096) at T=1 and T=0, CUDA events around
each call, with its dominant traffic: W_lm read once per position,
gamma * d * V * 2 bytes a call.  Prints one JSON line per measurement.
"""
from __future__ import annotations

import argparse
import json

import numpy as np

from . import synth


def _events():
    import torch
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def time_confidence(calls: int) -> None:
    import torch
    from . import dspark_confidence
    dev = torch.device("cuda", 0)
    for (R, g, d, V, rank) in [(128, 16, 4096, 151936, 256), (256, 16, 7168, 129280, 256)]:
        gen = torch.Generator(device=dev)
        gen.manual_seed(0)
        nb = max(2, (256 << 20) // (R * g * d * 2) + 1)  # rotating buffers, more bytes than L2
        hs = [torch.randn(R, g, d, device=dev, generator=gen).to(torch.bfloat16).view(torch.int16) for _ in range(nb)]
        W1 = (torch.randn(V, rank, device=dev, generator=gen) * 0.03).to(torch.bfloat16).view(torch.int16)
        w = torch.randn(d + rank, device=dev, generator=gen) * 0.02
        anchors = torch.randint(0, V, (R,), device=dev, dtype=torch.int32, generator=gen)
        tokens = torch.randint(0, V, (R, g), device=dev, dtype=torch.int32, generator=gen)
        c = torch.empty(R, g, device=dev)
        a = torch.empty(R, g, device=dev)
        ws = torch.zeros(256, dtype=torch.uint8, device=dev)
        for k in range(3):
            dspark_confidence(hs[k % nb], W1, w, anchors, tokens, c, a, ws)
        per_call = []
        for _ in range(5):
            e0, e1 = _events()
            e0.record()
            for k in range(calls):
                dspark_confidence(hs[k % nb], W1, w, anchors, tokens, c, a, ws)
            e1.record()
            torch.cuda.synchronize()
            per_call.append(e0.elapsed_time(e1) / calls)
        ms = float(np.median(per_call))
        print(json.dumps({"call": "dspark_confidence", "R": R, "gamma": g, "d": d, "ms": ms,
                          "h_GBps": R * g * d * 2 / (ms * 1e-3) / 1e9}), flush=True)


def time_verify(calls: int) -> None:
    import torch
    from .round import DeviceRound
    wl = synth.WORKLOADS["r128_g16_v151936"]
    W1, W2, w = synth.weights(wl)
    inp = synth.round_inputs(wl, 0)
    dr = DeviceRound(wl.R, wl.gamma, wl.V, wl.rank, wl.d)
    dr.set_weights(W1, W2, w)
    dr.set_round(inp.U, inp.h, inp.anchors, synth.sps_table(wl))
    dr.clear_status()
    dr.draft(1.0, wl.seed, 0)
    # target logits as the bench builds them: U + Markov bias of the drafted prefix + noise
    gen = torch.Generator(device=dr.device)
    gen.manual_seed(wl.seed * 1000)
    W1f = (dr.W1.to(torch.int32) << 16).view(torch.float32)
    W2f = (dr.W2.to(torch.int32) << 16).view(torch.float32)
    prev = torch.cat([dr.anchors.view(-1, 1).long(), dr.tokens[:, :-1].long()], dim=1)
    for r0 in range(0, wl.R, 16):
        r1 = min(wl.R, r0 + 16)
        bias = (W1f[prev[r0:r1].reshape(-1)] @ W2f).view(r1 - r0, wl.gamma, wl.V)
        noise = torch.randn((r1 - r0, wl.gamma + 1, wl.V), generator=gen, device=dr.device)
        dr.T[r0:r1, :wl.gamma] = dr.U[r0:r1] + bias + noise[:, :wl.gamma]
        dr.T[r0:r1, wl.gamma] = torch.randn((r1 - r0, wl.V), generator=gen, device=dr.device) * wl.u_std + noise[:, -1]
    dr.confidence()
    dr.schedule(0)
    torch.cuda.synchronize()
    for cs in (False, True):
        for _ in range(3):
            dr.verify(1.0, wl.seed, 0, c_star=cs)
        ts = []
        for _ in range(calls):
            e0, e1 = _events()
            e0.record()
            dr.verify(1.0, wl.seed, 0, c_star=cs)
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        print(json.dumps({"call": "dspark_verify", "c_star": cs, "verified_rows": int((dr.lens + 1).sum()),
                          "ms": float(np.median(ts)), "status": dr.status()}), flush=True)


def time_lmhead(calls: int) -> None:
    import torch
    from . import dspark_markov_draft_lmhead, lib
    wl = synth.WORKLOADS["r128_g16_v151936"]
    dev = torch.device("cuda", 0)
    W1, W2, _ = synth.weights(wl)
    W_lm = synth.lm_head_weight(wl)
    h = np.stack([synth.hidden(wl, 0, r) for r in range(wl.R)])
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    hd, Wl, W1d, W2d = t(h.view(np.int16)), t(W_lm.view(np.int16)), t(W1.view(np.int16)), t(W2.view(np.int16))
    ad = t(synth.anchors(wl, 0).astype(np.int32))
    tok = torch.empty((wl.R, wl.gamma), dtype=torch.int32, device=dev)
    pd = torch.empty((wl.R, wl.gamma), dtype=torch.float32, device=dev)
    lz = torch.empty_like(pd)
    ws = torch.zeros(lib().dspark_workspace_size(wl.R, wl.gamma, wl.V, wl.rank, wl.d), dtype=torch.uint8, device=dev)
    wlm_bytes = wl.gamma * wl.d * wl.V * 2
    for temperature in (1.0, 0.0):
        for _ in range(2):
            dspark_markov_draft_lmhead(hd, Wl, W1d, W2d, ad, temperature, wl.seed, 0, tok, pd, lz, ws)
        ts = []
        for _ in range(calls):
            e0, e1 = _events()
            e0.record()
            dspark_markov_draft_lmhead(hd, Wl, W1d, W2d, ad, temperature, wl.seed, 0, tok, pd, lz, ws)
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        ms = float(np.median(ts))
        print(json.dumps({"call": "dspark_markov_draft_lmhead", "temperature": temperature, "R": wl.R,
                          "gamma": wl.gamma, "V": wl.V, "d": wl.d, "ms": ms, "W_lm_bytes": wlm_bytes,
                          "W_lm_GBps": wlm_bytes / (ms * 1e-3) / 1e9,
                          "status": int(ws[:4].view(torch.int32).item())}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("what", choices=["confidence", "verify", "lmhead"])
    ap.add_argument("--calls", type=int, default=40)
    args = ap.parse_args(argv)
    if args.what == "confidence":
        time_confidence(args.calls)
    elif args.what == "lmhead":
        time_lmhead(args.calls)
    else:
        time_verify(args.calls)


if __name__ == "__main__":
    main()
