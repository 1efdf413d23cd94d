#!/usr/bin/env python
"""Benchmark of one DSpark speculative-decoding round on GB300.

A step is one whole round on the batch-128 long-block workload (R = 128
requests, gamma = 16 draft positions, V = 151936, rank 256, d = 4096,
temperature 1, early-stop scheduler on the page-2 SPS(B) table):
Markov draft -> confidence -> schedule -> verify, through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gpu|reference]

Prints one JSON line.  `value` = draft tokens sampled and verified per second
(R * gamma per round, all ranks) with inputs resident in HBM; `e2e` = the
same metric with the round's inputs copied from pinned host memory and the
results read back inside the timed region.  Under torchrun every rank runs
an independent replica on its own requests (weak scaling, no collective in
the data path); the time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "draft tokens sampled+verified/sec and achieved HBM GB/s vs GB300 peak, 1 GPU"
DEFAULT_WORKLOAD = "r128_g16_v151936"
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes per dspark_markov_draft call (one round's 16 positions) from the
# ncu capture summarised in profiles/; valid only for the draft kernel sources
# whose digest (draft_digest) is recorded with it.
NCU_DRAFT_TRAFFIC = {"digest": "d020ed141c19", "workload": "r128_g16_v151936", "bytes_per_call": 1377694720 + 17224192}


# ----------------------------------------------------------------------------- helpers
_C_TOKENS = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\\n])*"|\'(?:\\.|[^\'\\\n])*\'', re.S)


def code_text(src: str) -> str:
    """C/C++/CUDA source as the compiler sees it, up to layout: comments
    dropped (string and character literals kept), whitespace runs collapsed.
    Editing a comment or re-wrapping lines leaves it unchanged."""
    out = _C_TOKENS.sub(lambda m: " " if m.group(0)[0] == "/" else m.group(0), src)
    return " ".join(out.split())


def _digest(paths, code_only: bool = False) -> str:
    h = hashlib.sha1()
    for f in sorted(paths):
        with open(f, "rb") as fh:
            data = fh.read()
        if code_only:
            data = code_text(data.decode("utf-8")).encode("utf-8")
        h.update(os.path.basename(f).encode() + b"\0" + data)
    return h.hexdigest()[:12]


def kernel_digest() -> str:
    """Digest of every kernel source of the library."""
    return _digest(glob.glob(os.path.join(ROOT, "semi_autoregressive_speculative_gb300", "csrc", "*")))


def draft_digest() -> str:
    """Digest of the code (comments and layout aside) of the sources the draft
    kernel is compiled from."""
    csrc = os.path.join(ROOT, "semi_autoregressive_speculative_gb300", "csrc")
    names = ["markov_draft.cu", "common.h", "device.cuh", "search.cuh", "vocab_common.h"]
    return _digest([os.path.join(csrc, n) for n in names] + [os.path.join(ROOT, "include", "dspark.h")],
                   code_only=True)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Maximum of x over all ranks (identity on one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None) -> None:
    if world > 1:
        import torch.distributed as dist
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms while the
    timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.idx = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return self
        # the timed region starts only once the sampler is producing rows
        t0 = time.time()
        while time.time() - t0 < 5.0 and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except OSError:
            pass
        finally:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- CPU oracle (baseline)
_WEIGHTS = {}


def _weights(wl):
    from semi_autoregressive_speculative_gb300 import synth
    if wl.name not in _WEIGHTS:
        _WEIGHTS[wl.name] = synth.weights(wl)
    return _WEIGHTS[wl.name]


def oracle_sample(wl, requests, rnd: int = 0):
    """Time the CPU oracle on whole rounds of `requests` (inputs prepared
    outside the timed region).  Returns (seconds, tokens)."""
    import oracle
    from semi_autoregressive_speculative_gb300 import synth
    W1, W2, w = _weights(wl)
    inp = synth.round_inputs(wl, rnd, requests=requests)
    sps = synth.sps_table(synth.scaled(wl, R=len(requests), name=wl.name + "_sample"))
    t0 = time.perf_counter()
    tok, pd, lz = oracle.draft(inp.U, W1, W2, inp.anchors, wl.temperatures[0], wl.seed, rnd, request_ids=requests)
    c, a = oracle.confidence(inp.h, W1, w, inp.anchors, tok)
    mode = 2 if 2 in wl.modes else 0
    s = oracle.schedule(a, sps, mode)
    t1 = time.perf_counter()
    # target logits of the sample: harness work, outside the timed region
    T = np.empty((len(requests), wl.gamma + 1, wl.V), np.float32)
    for i, r in enumerate(requests):
        prevs = [int(inp.anchors[i])] + [int(x) for x in tok[i, :-1]]
        bias = np.stack([oracle.markov_bias(W1, W2, p) for p in prevs])
        T[i] = synth.compose_target(inp.U[i], bias, synth.target_noise(wl, rnd, r), synth.bonus_base(wl, rnd, r))
    t2 = time.perf_counter()
    oracle.verify(T, inp.U, W1, W2, inp.anchors, tok, s["lens"], wl.temperatures[0], wl.seed, rnd,
                  request_ids=requests)
    t3 = time.perf_counter()
    return (t1 - t0) + (t3 - t2), len(requests) * wl.gamma


def run_reference(args):
    rank, world, _ = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        if rank != 0:
            dist.barrier()
            return
    from semi_autoregressive_speculative_gb300 import synth
    import oracle
    oracle.build()
    wl = synth.WORKLOADS[args.workload]
    n = args.ref_sample_requests
    for i in range(args.warmup):
        oracle_sample(wl, [i % wl.R])
    times, toks = [], 0
    for i in range(args.steps):
        reqs = [(i * n + k) % wl.R for k in range(n)]
        t, k = oracle_sample(wl, reqs)
        times.append(t)
        toks += k
    value = toks / sum(times)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": wl.name, "R": wl.R, "gamma": wl.gamma, "V": wl.V, "rank": wl.rank, "d": wl.d},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"{n} request(s) of the workload per step: draft of all gamma positions, "
                                       f"confidence, schedule, verify; host has {os.cpu_count()} cores"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- GPU arm
def synth_target(dr, wl, rnd: int, seed: int):
    """Target logits on the device: U + Markov bias of the drafted prefix +
    noise; the bonus row a fresh U-distributed row + noise (harness work,
    torch ops, outside every timed region)."""
    import torch
    g = torch.Generator(device=dr.device)
    g.manual_seed(seed * 1000 + rnd)
    W1f = (dr.W1.to(torch.int32) << 16).view(torch.float32)
    W2f = (dr.W2.to(torch.int32) << 16).view(torch.float32)
    prev = torch.cat([dr.anchors.view(-1, 1).long(), dr.tokens[:, :-1].long()], dim=1)  # [R, gamma]
    std = torch.full((wl.R, 1, 1), wl.t_noise[0], device=dr.device)
    std[wl.R // 2:] = wl.t_noise[1]
    for r0 in range(0, wl.R, 16):
        r1 = min(wl.R, r0 + 16)
        bias = W1f[prev[r0:r1].reshape(-1)] @ W2f
        noise = torch.randn((r1 - r0, wl.gamma, wl.V), generator=g, device=dr.device) * std[r0:r1]
        dr.T[r0:r1, :wl.gamma] = dr.U[r0:r1] + bias.view(r1 - r0, wl.gamma, wl.V) + noise
        fresh = torch.randn((r1 - r0, wl.V), generator=g, device=dr.device) * wl.u_std
        dr.T[r0:r1, wl.gamma] = fresh + torch.randn((r1 - r0, wl.V), generator=g, device=dr.device) * std[r0:r1, 0]


def run_gpu(args):
    import torch
    rank, world, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    import semi_autoregressive_speculative_gb300 as pkg
    from semi_autoregressive_speculative_gb300 import build as pkg_build, synth
    from semi_autoregressive_speculative_gb300.round import DeviceRound
    if not os.path.exists(pkg.LIB_PATH):
        pkg_build.build()
    pkg.lib()

    wl = synth.WORKLOADS[args.workload]
    if args.gamma:  # smaller footprint of the same kernels (profiling captures)
        wl = synth.scaled(wl, gamma=args.gamma, name=f"{wl.name}_gamma{args.gamma}")
    temp = wl.temperatures[0]
    mode = 2 if 2 in wl.modes else 0
    seed, rnd = wl.seed, rank  # each rank: its own requests (round index = rank)
    W1, W2, w = synth.weights(wl)
    inp = synth.round_inputs(wl, rnd)
    dr = DeviceRound(wl.R, wl.gamma, wl.V, wl.rank, wl.d, device=device)
    dr.set_weights(W1, W2, w)
    dr.set_round(inp.U, inp.h, inp.anchors, synth.sps_table(wl))
    del inp
    dr.clear_status()
    dr.draft(temp, seed, rnd)
    synth_target(dr, wl, rnd, seed)
    torch.cuda.synchronize()

    calls = [lambda: dr.draft(temp, seed, rnd), lambda: dr.confidence(), lambda: dr.schedule(mode),
             lambda: dr.verify(temp, seed, rnd)]
    stream = torch.cuda.Stream(device=device)
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for f in calls:
            f()
    torch.cuda.synchronize()
    # one graph per call (for the per-call breakdown) and one for the whole round (the timed step)
    graphs = []
    for f in calls:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            f()
        graphs.append(g)
    round_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(round_graph, stream=stream):
        for f in calls:
            f()
    # verify with the optional analytic acceptance c*: reported beside the
    # breakdown, not part of the timed round
    cstar_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cstar_graph, stream=stream):
        dr.verify(temp, seed, rnd, c_star=True)
    # draft: a prologue kernel and one persistent kernel; confidence 1; schedule 1; verify 3 (greedy) or 5
    launches_per_step = 2 + 1 + 1 + (3 if temp == 0 else 5)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            round_graph.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, device)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            start.record(stream)
            for _ in range(args.steps):
                round_graph.replay()
            end.record(stream)
        torch.cuda.synchronize()
    barrier(world, device)
    elapsed = start.elapsed_time(end) / 1e3
    t_max = max_over_ranks(elapsed, world, device)
    # per-call breakdown, outside the timed region: each call's graph replayed on its own
    n_bd = max(3, min(args.steps, 50))
    per_call = []
    with torch.cuda.stream(stream):
        for g in graphs + [cstar_graph]:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n_bd):
                g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            per_call.append(e0.elapsed_time(e1) / n_bd)  # ms
    status = dr.status()
    lens_h = dr.lens.cpu().numpy()
    nacc_h = dr.n_accept.cpu().numpy()

    R, g, V, rk, d = wl.R, wl.gamma, wl.V, wl.rank, wl.d
    tokens_per_step = R * g
    value = tokens_per_step * world * args.steps / t_max
    # algorithmic bytes of one dspark_markov_draft call: U read once, W2 once,
    # the gathered W1 rows (tensor-core pass and sampler), the outputs
    draft_bytes = R * g * V * 4 + rk * V * 2 + 2 * R * g * rk * 2 + 12 * R * g
    peak, peak_src = measured_peaks()
    achieved = draft_bytes / (per_call[0] / 1e3) / 1e9
    # whole-round algorithmic bytes: the draft's, h and the confidence's W1
    # rows, the target rows verify reads, and the residual recompute of the
    # rejected rows (their U and T rows, W2 once)
    rows_read = int((lens_h + 1).sum())
    n_rej = int((nacc_h < lens_h).sum()) if temp > 0 else 0
    round_bytes = (draft_bytes + R * g * d * 2 + R * g * rk * 2 + rows_read * V * 4 + n_rej * V * 8 +
                   (rk * V * 2 if n_rej else 0))
    round_gbs = round_bytes / (t_max / args.steps) / 1e9
    # c* re-reads the U and T rows of every verified position with a draft
    # distribution (W2 once) on top of the target-row statistics
    cstar_rows = int(np.minimum(lens_h + 1, g).sum()) if temp > 0 else 0
    cstar_bytes = rows_read * V * 4 + cstar_rows * V * 8 + (rk * V * 2 if cstar_rows else 0)
    digest = kernel_digest()
    # the recorded DRAM bytes belong to one full call of the workload they were captured on
    traffic = (NCU_DRAFT_TRAFFIC["bytes_per_call"]
               if NCU_DRAFT_TRAFFIC["digest"] == draft_digest() and wl.name == NCU_DRAFT_TRAFFIC["workload"] else None)

    # ------------------------------------------------------------- end to end (host buffers)
    # Every step brings the round's inputs in from pinned host memory and reads
    # its results back.  Verify reads only target rows 0..lens[r] of request r,
    # and those lengths are decided on the device by the scheduler: the step
    # brings in just those rows with dspark_load_verified_rows (the SMs read
    # them from the mapped host memory, driven by the lengths on the device),
    # as a serving loop that evaluates only the scheduled positions would.  U
    # and h, the bulk of the bytes, are double-buffered: the copy engines bring
    # in the next step's U and h while this step computes.  The host link
    # (about 210 GB/s on this part) is the bound.
    e2e = None
    if not args.no_e2e:
        hU = torch.empty(dr.U.shape, dtype=dr.U.dtype, pin_memory=True)
        hT = torch.empty(dr.T.shape, dtype=dr.T.dtype, pin_memory=True)
        hh = torch.empty(dr.h.shape, dtype=dr.h.dtype, pin_memory=True)
        hU.copy_(dr.U)
        hT.copy_(dr.T)
        hh.copy_(dr.h)
        outs = [dr.tokens, dr.n_accept, dr.next_token]
        hout = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
        n_e2e = max(1, min(args.steps, 10))
        u_bufs = [dr.U, torch.empty_like(dr.U)]
        h_bufs = [dr.h, torch.empty_like(dr.h)]
        copy_stream = torch.cuda.Stream(device=device)

        def issue_inputs(k):
            # step k's U and h into buffers k % 2, whose last reader (step k - 2) has finished
            ev = torch.cuda.Event()
            with torch.cuda.stream(copy_stream):
                u_bufs[k % 2].copy_(hU, non_blocking=True)
                h_bufs[k % 2].copy_(hh, non_blocking=True)
                ev.record(copy_stream)
            return ev

        def e2e_step(k, n, ready):
            dr.U, dr.h = u_bufs[k % 2], h_bufs[k % 2]
            stream.wait_event(ready)
            ready_next = issue_inputs(k + 1) if k + 1 < n else None  # overlaps this step
            calls[0]()  # draft
            calls[1]()  # confidence
            calls[2]()  # schedule
            dr.load_target_rows(hT)
            calls[3]()  # verify
            for o, ho in zip(outs, hout):
                ho.copy_(o, non_blocking=True)
            stream.synchronize()
            return ready_next

        def run_steps(n):
            ready = issue_inputs(0)
            for k in range(n):
                with torch.cuda.stream(stream):
                    ready = e2e_step(k, n, ready)
            torch.cuda.synchronize()

        run_steps(2)  # untimed
        barrier(world, device)
        t0 = time.perf_counter()
        run_steps(n_e2e)
        t_e2e = max_over_ranks(time.perf_counter() - t0, world, device)
        dr.U, dr.h = u_bufs[0], h_bufs[0]
        # every step drafts the same round, so it admits the same rows_read target rows
        e2e = {"value": tokens_per_step * world * n_e2e / t_e2e, "unit": "tokens/s",
               "h2d_bytes_per_step": int(hU.numel() * 4 + hh.numel() * 2 + rows_read * V * 4),
               "d2h_bytes_per_step": int(sum(o.numel() * o.element_size() for o in outs)),
               "steps": n_e2e,
               "note": "U and h in every step, by the copy engines, double-buffered (the next step's U and h "
                       "come in while this step computes); the target rows of the verified positions only, read "
                       "from pinned host memory by dspark_load_verified_rows with the lengths on the device"}

    # ------------------------------------------------------------- CPU oracle on a bounded sample
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        reqs = list(range(args.cpu_sample_requests))
        secs, toks = oracle_sample(wl, reqs)
        cpu = {"value": toks / secs, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"{len(reqs)} of {R} requests, one whole round each (draft of {g} positions, "
                         f"confidence, schedule, verify); single-threaded C oracle, host has "
                         f"{os.cpu_count()} cores; {secs:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * t_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": wl.name, "R": R, "gamma": g, "V": V, "rank": rk, "d": d, "temperature": temp,
                       "scheduler": ["early_stop", "top_k", "fixed"][mode], "parallelism": f"replicas{world}",
                       "l2": f"inputs larger than L2: U {R * g * V * 4 / 1e9:.2f} GB and T "
                             f"{R * (g + 1) * V * 4 / 1e9:.2f} GB per round",
                       "timing": "one CUDA graph per round (draft, confidence, schedule, verify); breakdown from each call's own graph"},
            "roofline": {"kernel": "k_markov_draft (dspark_markov_draft: one persistent launch, all gamma positions)",
                         "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "peak_source": peak_src,
                         "algorithmic_bytes": draft_bytes, "ms_per_call": per_call[0]},
            "breakdown_ms": {"draft": per_call[0], "confidence": per_call[1], "schedule": per_call[2],
                             "verify": per_call[3]},
            "verify_c_star": {"ms": per_call[4], "rows": cstar_rows, "algorithmic_bytes": cstar_bytes,
                              "achieved": cstar_bytes / (per_call[4] / 1e3) / 1e9, "unit": "GB/s",
                              "note": "dspark_verify with the optional c* output; outside the timed round"},
            "round": {"algorithmic_bytes": round_bytes, "achieved": round_gbs, "unit": "GB/s",
                      "frac": round_gbs / peak, "verified_rows": rows_read, "rejected_rows": n_rej,
                      "admitted_positions": int(lens_h.sum())},
            "clocks": clk.summary(),
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "cpu_baseline": cpu,
            "status_word": status,
            "kernel_digest": digest,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--gamma", type=int, default=0,
                    help="override the workload's draft length (smaller profiling cases only)")
    ap.add_argument("--cpu-sample-requests", type=int, default=16,
                    help="requests in the CPU-oracle baseline sample of the GPU arm")
    ap.add_argument("--ref-sample-requests", type=int, default=2,
                    help="requests per step of the reference (CPU oracle) arm")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
