"""Per-position phase breakdown of the Markov draft kernel (a profiling tool).

    python -m semi_autoregressive_speculative_gb300.draft_trace \\
        [--workload r128_g16_v151936] [--temperature 1.0] [--calls 5] [--lib PATH]

Builds ``lib/libdspark_trace.so`` (build.py --trace: the same sources with the
draft kernel's global-timer stamps compiled in), runs dspark_markov_draft on the
workload's seeded synthetic inputs a few times and prints, for the last call,
the median time of every phase of a draft position: over CTAs for the per-CTA
phases and over positions 1 .. gamma-2.  The stamps are the kernel's
``TraceEvent`` list in csrc/markov_draft.cu.  The traced build adds a handful
of global stores per position; the product library has none of them.
"""
from __future__ import annotations

import argparse
import ctypes
import json

import numpy as np

from . import build as pkg_build
from . import synth

EVENTS = ["a_ready", "first_acc", "tiles_done", "entry", "poll_done", "chunk_found", "fine_loaded", "slab_issued",
          "slab_landed", "picked", "published", "ready_seen", "copy_first", "copy_third", "start", "end", "launch",
          "pro_start", "pro_end"]
K_MTILE, K_TILE_N, K_MAX_CHUNKS = 128, 64, 1024


def _lib(path=None):
    L = ctypes.CDLL(path or pkg_build.build(trace=True))
    P, I, F, U64, U32, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint64, ctypes.c_uint32,
                             ctypes.c_size_t)
    L.dspark_workspace_size.restype = SZ
    L.dspark_workspace_size.argtypes = [I, I, I, I, I]
    L.dspark_markov_draft.restype = I
    L.dspark_markov_draft.argtypes = [P, P, P, P, I, I, I, I, F, U64, U32, P, P, P, P, SZ, P]
    L.dspark_draft_trace_buffer.restype = I
    L.dspark_draft_trace_buffer.argtypes = [P, SZ]
    return L


def grid_size(R: int, V: int, sm_count: int) -> int:
    """CTAs of one draft launch: contiguous vocabulary chunks x M-tiles (the
    host rule of csrc/markov_draft.cu vocab_chunks)."""
    n_m = -(-R // K_MTILE)
    n_tiles = -(-V // K_TILE_N)
    chunks = max(1, min(sm_count // n_m, n_tiles, K_MAX_CHUNKS))
    return chunks * n_m


def phases(tr: np.ndarray, R: int) -> dict:
    """Median phase durations (µs) from stamps tr [gamma, n_ctas, len(EVENTS)] (ns)."""
    g, n, _ = tr.shape
    e = {name: tr[:, :, i].astype(np.float64) for i, name in enumerate(EVENTS)}
    samplers = np.arange(min(R, n))  # CTA c samples request c first
    js = range(1, g - 1)
    us = lambda x: float(np.median(x)) / 1e3  # noqa: E731
    out = {
        "period": us([e["a_ready"][j + 1] - e["a_ready"][j] for j in js]),
        "a_ready_to_first_acc": us([e["first_acc"][j] - e["a_ready"][j] for j in js]),
        "tiles": us([e["tiles_done"][j] - e["first_acc"][j] for j in js]),
        "tiles_end_spread": us([e["tiles_done"][j].max() - e["tiles_done"][j].min() for j in js]),
        "tiles_end_last_minus_median": us([e["tiles_done"][j].max() - np.median(e["tiles_done"][j]) for j in js]),
        "entry_publish": us([e["entry"][j] - e["tiles_done"][j] for j in js]),
        "poll_after_last_entry": us([e["poll_done"][j][samplers] - e["entry"][j].max() for j in js]),
        "merge_and_chunk_search": us([e["chunk_found"][j][samplers] - e["poll_done"][j][samplers] for j in js]),
        "fine_load": us([e["fine_loaded"][j][samplers] - e["chunk_found"][j][samplers] for j in js]),
        "subtile_search_and_slab_issue": us([e["slab_issued"][j][samplers] - e["fine_loaded"][j][samplers] for j in js]),
        "slab_land": us([e["slab_landed"][j][samplers] - e["slab_issued"][j][samplers] for j in js]),
        "pick": us([e["picked"][j][samplers] - e["slab_landed"][j][samplers] for j in js]),
        "publish": us([e["published"][j][samplers] - e["picked"][j][samplers] for j in js]),
        "ready_seen_after_last_publish": us([e["ready_seen"][j + 1] - e["published"][j][samplers].max() for j in js]),
        "a_store": us([e["a_ready"][j + 1] - e["ready_seen"][j + 1] for j in js]),
        # the chain from the last CTA's last tile to the next position's A operand, on the slowest path
        "chain_last_tile_to_next_a": us([e["a_ready"][j + 1].max() - e["tiles_done"][j].max() for j in js]),
        "last_entry_to_last_publish": us([e["published"][j][samplers].max() - e["entry"][j].max() for j in js]),
        # the copier's lead: when the next position's first and third U pairs were in tensor memory,
        # relative to this position's last tile (negative: before it)
        "next_copy_first_after_tiles": us([e["copy_first"][j + 1] - e["tiles_done"][j] for j in js]),
        "next_copy_third_after_tiles": us([e["copy_third"][j + 1] - e["tiles_done"][j] for j in js]),
    }
    # the call outside the position periods: set-up to position 0's A operand, and the last position's
    # publish to the last CTA's exit
    start, end = e["start"][0], e["end"][0]
    out["kernel_span"] = float(end.max() - start.min()) / 1e3
    out["setup_to_first_a"] = us(e["a_ready"][0] - start.min())
    out["start_spread"] = float(start.max() - start.min()) / 1e3  # CTAs' set-up done, last minus first
    out["setup_to_first_a_same_cta"] = us(e["a_ready"][0] - start)
    # before the kernel: the prologue launch, the gap to the draft's first instruction, the draft's set-up
    launch, ps, pe = e["launch"][0], e["pro_start"][0], e["pro_end"][0]
    out["prologue_span"] = float(pe.max() - ps.min()) / 1e3
    out["prologue_end_to_first_launch"] = float(launch.min() - pe.max()) / 1e3
    out["launch_spread"] = float(launch.max() - launch.min()) / 1e3
    out["launch_to_setup_done"] = us(start - launch)
    out["first_position_period"] = us(e["a_ready"][1] - e["a_ready"][0])
    out["last_position_a_to_end"] = float(end.max() - np.median(e["a_ready"][g - 1])) / 1e3
    return out


def main(argv=None):
    import torch
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="r128_g16_v151936")
    ap.add_argument("--temperature", type=float, default=None)
    ap.add_argument("--calls", type=int, default=5)
    ap.add_argument("--lib", default=None, help="a library built with the trace stamps (default: build lib/libdspark_trace.so)")
    args = ap.parse_args(argv)
    wl = synth.WORKLOADS[args.workload]
    temp = wl.temperatures[0] if args.temperature is None else args.temperature
    L = _lib(args.lib)
    dev = torch.device("cuda", 0)
    W1, W2, _ = synth.weights(wl)
    inp = synth.round_inputs(wl, 0)
    U = torch.from_numpy(inp.U).to(dev)
    W1d = torch.from_numpy(W1.view(np.int16)).to(dev)
    W2d = torch.from_numpy(W2.view(np.int16)).to(dev)
    anchors = torch.from_numpy(inp.anchors).to(dev)
    R, g, V, rank = wl.R, wl.gamma, wl.V, wl.rank
    tokens = torch.empty((R, g), dtype=torch.int32, device=dev)
    pd = torch.empty((R, g), dtype=torch.float32, device=dev)
    lz = torch.empty((R, g), dtype=torch.float32, device=dev)
    ws = torch.zeros(L.dspark_workspace_size(R, g, V, rank, wl.d), dtype=torch.uint8, device=dev)
    n_ctas = grid_size(R, V, torch.cuda.get_device_properties(dev).multi_processor_count)
    trace = torch.zeros((g, n_ctas, len(EVENTS)), dtype=torch.int64, device=dev)
    L.dspark_draft_trace_buffer(trace.data_ptr(), trace.numel() * 8)
    stream = torch.cuda.current_stream().cuda_stream
    times = []
    for _ in range(args.calls):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        rc = L.dspark_markov_draft(U.data_ptr(), W1d.data_ptr(), W2d.data_ptr(), anchors.data_ptr(), R, g, V, rank,
                                   float(temp), wl.seed, 0, tokens.data_ptr(), pd.data_ptr(), lz.data_ptr(),
                                   ws.data_ptr(), ws.numel(), stream)
        e1.record()
        torch.cuda.synchronize()
        if rc != 0:
            raise RuntimeError(f"dspark_markov_draft returned {rc}")
        times.append(e0.elapsed_time(e1))
    status = int(ws[:4].view(torch.int32).item())
    tr = trace.cpu().numpy()
    res = {"workload": wl.name, "temperature": temp, "ctas": n_ctas, "status": status,
           "ms_per_call_traced": float(np.median(times)), "phases_us": phases(tr, R)}
    print(json.dumps(res, indent=1))


if __name__ == "__main__":
    main()
