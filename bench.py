#!/usr/bin/env python3
"""Benchmark: chunked Gated DeltaNet forward + backward on GB300.

One step = one forward (o, S_T) and one backward (dq, dk, dv, dg, dbeta) of the
H=32, T=8192, d=128 bf16 prefill workload through the C ABI, inputs resident in
HBM.  By default the pair is gdn_chunk_fwd_save + gdn_chunk_bwd_saved (the
forward keeps its per-chunk states and WY tiles for the backward); --recompute
times gdn_chunk_fwd + gdn_chunk_bwd, and each run also reports the other pair.
Prints ONE JSON line (rank 0).  See --help for the options.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gb300|reference]

Timing: W untimed warm-up steps; K timed steps, each bracketed by CUDA events on
the launch stream, with an L2 flush (a 256 MB write) before every step that is
outside the events; barrier + synchronize around the timed loop; max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN chunked fwd+bwd tokens/s (bf16, d=128) on 1 GB300; % of HBM roofline"
DEFAULT_WORKLOAD = "prefill_h32_t8192"


# ----------------------------------------------------------------------------- accounting
def algorithmic_bytes(w, x):
    """Bytes the method must move (per call), per the roofline accounting:
    forward 2*(dk+dk+dv)*e + 8 + dv*e per token-head (q, k, v, g, beta in; o out) plus
    4*d^2 per (sequence, head) for S0 in / S_T out; backward q, k, v, dO, g, beta in and
    dq, dk, dv, dg, dbeta out plus the state terms."""
    e = 2 if x["dtype"] == "bf16" else 4
    D = x["D"]
    tokens = x["q"].shape[0] * x["q"].shape[1]
    th = tokens * x["H"]
    sh = x["N"] * x["H"]
    st = 4 * D * D
    fwd = th * (3 * D * e + 8 + D * e) + sh * st * ((x["S0"] is not None) + 1)
    bwd = th * (4 * D * e + 8 + 3 * D * e + 8) + sh * st * ((x["S0"] is not None) * 2 + (x["dST"] is not None))
    per_kernel = {
        "fwd_chunk": fwd,
        "fwd_states": th * (3 * D * e + 8),        # q, k, v, g, beta in (state copies are workspace)
        "bwd_chain": th * (3 * D * e + 8),         # q, k, dO, g, beta in
        "bwd_local": th * (4 * D * e + 8 + 3 * D * e + 8),
    }
    return fwd, bwd, per_kernel


# ----------------------------------------------------------------------------- multi-rank host logic
def replica_seed(seed, rank):
    """Each rank runs its own replica of the workload, drawn from its own seed."""
    return seed + 1000 * rank


def max_over_ranks(local_ms, world, device=None):
    """The job's time is the slowest rank's: all-reduce MAX over the process group."""
    import torch
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(total_ms, world, tokens_per_rank_step, steps):
    """Whole-job tokens/s: `world` replicas each process `tokens_per_rank_step` per step."""
    return world * tokens_per_rank_step * steps / (total_ms / 1000.0)


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu capture,
# keyed by (profiler name, workload); valid only while the kernel's translation unit (its .cu file and
# the local headers it includes, transitively) hashes to the value recorded with it (otherwise the
# roofline reports traffic null).  Summaries: profiles/*.md.
NCU_TRAFFIC = {
    ("bwd_local", "prefill_h32_t8192"): (1022568192, "bwd_local_tc.cu", "f974d11495cedf5e"),
    ("fwd_chunk", "prefill_h32_t8192"): (599764224, "fwd_tc.cu", "1f89580d4ef10f85"),
    ("fwd_prep", "prefill_h32_t8192"): (513900800, "fwd_prep_tc.cu", "40c0954d21fe6409"),
    ("bwd_chain", "prefill_h32_t8192"): (537678080, "bwd_chain_tc.cu", "ec98eaa20e34262a"),
}


def kernel_sources(src):
    """The files of a kernel's translation unit: src and the local headers it includes, transitively."""
    import re
    csrc = os.path.join(ROOT, "gated_deltanet_linear_15_gb300", "csrc")
    seen, todo = set(), [src]
    while todo:
        f = todo.pop()
        if f in seen:
            continue
        seen.add(f)
        with open(os.path.join(csrc, f)) as fh:
            todo += re.findall(r'^\s*#include "([^"]+)"', fh.read(), flags=re.M)
    return sorted(seen)


def source_digest(src):
    import hashlib
    m = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_deltanet_linear_15_gb300", "csrc")
    for f in kernel_sources(src):
        m.update(f.encode())
        with open(os.path.join(csrc, f), "rb") as fh:
            m.update(fh.read())
    return m.hexdigest()[:16]


def measured_traffic(kernel, workload):
    ent = NCU_TRAFFIC.get((kernel, workload))
    if ent is None:
        return None
    nbytes, src, digest = ent
    try:
        return nbytes if source_digest(src) == digest else None
    except OSError:
        return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1901.0)), "measured"
    return 6800.0, 1900.0, "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4) if s[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples)}


# ----------------------------------------------------------------------------- CPU oracle legs
def cpu_oracle_sample(wname, heads=None, tokens=None):
    """Time the fp64 oracle (fwd + bwd) on a bounded sample of the workload: the
    first `heads` heads (default: one per core) over `tokens` tokens per sequence.
    Returns (tokens/s scaled to the whole workload's head count, cores, description)."""
    import torch

    import oracle
    from gdn_inputs import WORKLOADS, make_inputs
    w = WORKLOADS[wname]
    cores = os.cpu_count() or 1
    Hs = min(w.H, heads or cores)
    if not w.T:  # packed variable-length batch: the drawn lengths (~135k tokens), on fewer heads
        Hs = max(1, Hs // 4)
    T = tokens or (w.T if w.T else 4096)
    x = make_inputs(w, "cpu", H=Hs, T=T, B=1)
    T = x["q"].shape[0] * x["q"].shape[1]  # tokens actually in the sample
    t0 = time.perf_counter()
    oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], scale=x["scale"], l2norm=x["l2norm"],
               nthreads=cores)
    oracle.bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["dO"], x["S0"], None, scale=x["scale"],
               l2norm=x["l2norm"], nthreads=cores)
    dt = time.perf_counter() - t0
    # the workload's tokens/s: T tokens of all H heads cost H/Hs times the sample
    tps = T * (Hs / w.H) / dt
    return tps, min(cores, Hs * x["N"]), f"fwd+bwd of {Hs} of {w.H} heads x {T} tokens, {dt:.2f} s", dt, Hs / w.H


def run_reference(args):
    """--impl reference: the CPU oracle as it stands, on the host cores (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    tps_all, dts = [], []
    desc, cores, frac = "", 1, 1.0
    from gdn_inputs import WORKLOADS
    w = WORKLOADS[args.workload]
    for i in range(args.warmup + args.steps):
        tps, cores, desc, dt, frac = cpu_oracle_sample(args.workload, tokens=args.ref_tokens)
        if i >= args.warmup:
            tps_all.append(tps)
            dts.append(dt)
    value = statistics.median(tps_all)
    tokens_per_step = (w.B * w.T) if w.T else 135168
    # Each step is a bounded sample of the workload (a fraction of its heads); ms_per_step is the
    # sample's measured wall time, value the workload-equivalent throughput (sample tokens x head
    # fraction / time), and the whole-workload time per step it implies is given beside it.
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000.0 * statistics.median(dts), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "sampled": True, "sample_head_fraction": round(frac, 4), "timed_seconds": round(sum(dts), 3),
            "workload_ms_per_step_equivalent": 1000.0 * tokens_per_step / value,
            "config": {"workload": args.workload, "B": w.B, "T": w.T, "H": w.H, "d": w.D},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- segment-length sweep
def run_sweep(args, g, x, dev):
    """Saved-context fwd + bwd timed per segment length (CUDA events around each call, 256 MB L2 flush
    before every step, outside the events), with the mean time of the two recurrent passes (each
    bracketed alone over K further steps) and the library's own estimate for the plan
    (gdn_plan_estimate).  One JSON line per plan."""
    import torch
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    N, H, D = x["N"], x["H"], x["D"]
    o = torch.empty_like(x["v"])
    ST = torch.empty(N, H, D, D, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"])
    dg, db = torch.empty_like(x["g"]), torch.empty_like(x["beta"])
    dS0 = torch.empty_like(x["S0"]) if x["S0"] is not None else None
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    time.sleep(0.3)
    for spec in args.sweep_seg_chunks.split(","):
        L, F = (int(v) for v in spec.split(":")) if ":" in spec else (int(spec), 0)
        shape = g.make_shape(x["q"], x["v"], cu_seqlens=x["cu_seqlens"], scale=x["scale"], l2norm=x["l2norm"],
                             seg_chunks=L, seg_first=F)
        plan = g.gdn_plan_query(shape)
        est = g.gdn_plan_estimate(shape)
        ws_bytes = max(g.gdn_fwd_workspace_size(shape), g.gdn_bwd_saved_workspace_size(shape))
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        saved_bytes = g.gdn_saved_size(shape)
        saved = torch.empty(max(saved_bytes, 256), dtype=torch.uint8, device=dev)

        def fwd():
            rc = g.gdn_chunk_fwd_save(shape, x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], o, ST, saved, ws,
                                      saved_bytes, ws_bytes, stream)
            assert rc == 0, g._lib.last_error()

        def bwd():
            rc = g.gdn_chunk_bwd_saved(shape, x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], x["dO"], x["dST"],
                                       dq, dk, dv, dg, db, dS0, saved, ws, saved_bytes, ws_bytes, stream)
            assert rc == 0, g._lib.last_error()

        for _ in range(args.warmup):
            flush.zero_()
            fwd()
            bwd()
        # the recurrent passes, each bracketed alone (the other launches keep their overlap) over K steps
        kern = {}
        for name in ("fwd_chunk", "bwd_chain"):
            g.gdn_profile_report(reset=True)
            g.gdn_profile_only(name)
            g.gdn_profile_enable(True)
            for _ in range(args.steps):
                flush.zero_()
                fwd()
                bwd()
            torch.cuda.synchronize()
            g.gdn_profile_enable(False)
            kern.update(g.gdn_profile_report(reset=True))
        g.gdn_profile_only(None)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        torch.cuda.synchronize()
        for e in evs:
            flush.zero_()
            e[0].record(stream)
            fwd()
            e[1].record(stream)
            bwd()
            e[2].record(stream)
        torch.cuda.synchronize()
        fwd_ms = statistics.median(a.elapsed_time(b) for a, b, c in evs)
        bwd_ms = statistics.median(b.elapsed_time(c) for a, b, c in evs)
        print(json.dumps({"sweep": args.workload, "seg_chunks_requested": L, "seg_first": F,
                          "seg_chunks": plan["seg_chunks"],
                          "max_segments": plan["max_segments"], "fwd_ms": round(fwd_ms, 4),
                          "bwd_ms": round(bwd_ms, 4), "step_ms": round(fwd_ms + bwd_ms, 4),
                          "estimate_us": est,
                          "kernels_ms": {k: round(ms / c, 4) for k, (c, ms) in kern.items()}}), flush=True)
        del ws, saved
    print(json.dumps({"sweep_clocks": clocks.stop()}), flush=True)
    return 0


# ----------------------------------------------------------------------------- decode arm
def run_decode(args):
    """gdn_recurrent_fwd on B sequences x T tokens (H=32, d=128, bf16, fp32 state updated in place).
    The step is HBM-bound on the state: algorithmic bytes = state read + write (2 x 4 d^2 per
    (sequence, head)) + q, k, v, o (4 x 2 d per token-head) + g, beta (8 per token-head)."""
    import torch

    import __graft_entry__
    __graft_entry__.build_library()
    import gated_deltanet_linear_15_gb300 as g
    from gdn_inputs import make_inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    B, T, H, D = args.decode_batch, args.decode_tokens, 32, 128
    x = make_inputs("prefill_h32_t8192", dev, T=T, B=B, H=H, with_S0=True, seed=101)
    S = x["S0"].clone()
    o = torch.empty_like(x["v"])
    shape = g.make_shape(x["q"], x["v"], scale=x["scale"], l2norm=x["l2norm"])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        rc = g.gdn_recurrent_fwd(shape, x["q"], x["k"], x["v"], x["g"], x["beta"], S, o, S, stream)
        assert rc == 0, g._lib.last_error()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = [a.elapsed_time(b) for a, b in evs]
    step_ms = statistics.median(ms)
    hbm_peak, _, peak_kind = load_peaks()
    nbytes = B * H * 2 * 4 * D * D + B * T * H * (4 * 2 * D + 8)
    ach = nbytes / (step_ms / 1000.0) / 1e9
    line = {"metric": "GDN recurrent decode tokens/s (bf16, d=128, fp32 state) on 1 GB300",
            "value": B * T / (step_ms / 1000.0), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded gdn_inputs)",
            "config": {"workload": f"decode_b{B}_h{H}_t{T}", "B": B, "T": T, "H": H, "d": D,
                       "l2": "256 MB flush before every step, outside the events"},
            "roofline": {"bound": "hbm", "kernel": "recurrent", "achieved": round(ach, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(ach / hbm_peak, 4), "peak_kind": peak_kind, "traffic": None,
                         "algorithmic_bytes_per_launch": nbytes},
            "gpu_launches": args.steps, "clocks": clk}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm
def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-tokens", type=int, default=None, help="tokens per sequence in the reference sample")
    ap.add_argument("--seg-chunks", type=int, default=0)
    ap.add_argument("--sweep-seg-chunks", default="",
                    help="comma-separated segment lengths L or L:F (F = the first segment's length; 0 = the "
                         "automatic plan): time the saved-context pair for each and print one JSON line per "
                         "plan instead of the bench line")
    ap.add_argument("--recompute", action="store_true",
                    help="time the stateless pair (the backward recomputes the chunk states and WY tiles) "
                         "instead of the saved-context pair")
    ap.add_argument("--decode", action="store_true",
                    help="time the token-by-token decode entry point instead (B sequences x T tokens)")
    ap.add_argument("--decode-batch", type=int, default=64)
    ap.add_argument("--decode-tokens", type=int, default=1)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.decode:
        return run_decode(args)

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    # CPU baseline first (before heavy GPU work), rank 0 at N=1 only
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, cores, desc, _, _ = cpu_oracle_sample(args.workload)
        cpu = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc}

    import __graft_entry__
    __graft_entry__.build_library()
    import gated_deltanet_linear_15_gb300 as g
    from gdn_inputs import WORKLOADS, make_inputs

    w = WORKLOADS[args.workload]
    x = make_inputs(w, dev, seed=replica_seed(w.seed, rank))
    if args.sweep_seg_chunks:
        return run_sweep(args, g, x, dev)
    shape = g.make_shape(x["q"], x["v"], cu_seqlens=x["cu_seqlens"], scale=x["scale"], l2norm=x["l2norm"],
                         seg_chunks=args.seg_chunks)
    plan = g.gdn_plan_query(shape)
    ws_bytes = max(g.gdn_fwd_workspace_size(shape), g.gdn_bwd_workspace_size(shape))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    saved_bytes = g.gdn_saved_size(shape)
    saved = torch.empty(max(saved_bytes, 256), dtype=torch.uint8, device=dev)
    o = torch.empty_like(x["v"])
    N, H, D = x["N"], x["H"], x["D"]
    ST = torch.empty(N, H, D, D, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"])
    dg, db = torch.empty_like(x["g"]), torch.empty_like(x["beta"])
    dS0 = torch.empty_like(x["S0"]) if x["S0"] is not None else None
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    # One training step of the layer: the forward (o, S_T) then the backward (all gradients), both from
    # the inputs.  Saved-context pair (default): the forward also leaves its per-chunk states and WY
    # tiles in `saved` and the backward reads them; --recompute: the backward rederives them.
    def fwd_call(q, k, v, gg, beta, o_, recompute, st_=None):
        st_ = ST if st_ is None else st_
        if recompute:
            return g.gdn_chunk_fwd(shape, q, k, v, gg, beta, x["S0"], o_, st_, ws, ws_bytes, stream)
        return g.gdn_chunk_fwd_save(shape, q, k, v, gg, beta, x["S0"], o_, st_, saved, ws, saved_bytes, ws_bytes,
                                    stream)

    def bwd_call(q, k, v, gg, beta, dO, outs, recompute):
        ds0 = outs[5] if len(outs) > 5 else dS0
        a = (shape, q, k, v, gg, beta, x["S0"], dO, x["dST"], outs[0], outs[1], outs[2], outs[3], outs[4], ds0)
        if recompute:
            return g.gdn_chunk_bwd(*a, ws, ws_bytes, stream)
        return g.gdn_chunk_bwd_saved(*a, saved, ws, saved_bytes, ws_bytes, stream)

    def fwd(recompute=args.recompute):
        rc = fwd_call(x["q"], x["k"], x["v"], x["g"], x["beta"], o, recompute)
        assert rc == 0, g._lib.last_error()

    def bwd(recompute=args.recompute):
        rc = bwd_call(x["q"], x["k"], x["v"], x["g"], x["beta"], x["dO"], (dq, dk, dv, dg, db), recompute)
        assert rc == 0, g._lib.last_error()

    for _ in range(args.warmup):
        flush.zero_()
        fwd()
        bwd()
    torch.cuda.synchronize()

    # Per-kernel table: one pass of K steps with every launch bracketed by events (untimed).  The timed
    # loop below brackets only the dominant kernel, so its events add nothing to the other launches.
    g.gdn_profile_report(reset=True)
    g.gdn_profile_only(None)
    g.gdn_profile_enable(True)
    for _ in range(args.steps):
        flush.zero_()
        fwd()
        bwd()
    torch.cuda.synchronize()
    g.gdn_profile_enable(False)
    kern = g.gdn_profile_report(reset=True)
    dom = max(kern, key=lambda k: kern[k][1]) if kern else None

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    g.gdn_profile_only(dom)
    g.gdn_profile_enable(True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        fwd()
        evs[i][1].record(stream)
        bwd()
        evs[i][2].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    g.gdn_profile_enable(False)
    g.gdn_profile_only(None)
    clk = clocks.stop()
    live = g.gdn_profile_report(reset=True)  # the dominant kernel's launches inside the timed loop
    fwd_ms = [a.elapsed_time(b) for a, b, c in evs]
    bwd_ms = [b.elapsed_time(c) for a, b, c in evs]
    step_ms = sum(fwd_ms) + sum(bwd_ms)
    total_ms = max_over_ranks(step_ms, world, dev)
    tokens_per_step = x["q"].shape[0] * x["q"].shape[1]
    value = job_throughput(total_ms, world, tokens_per_step, args.steps)

    # ---- roofline of the dominant kernel, from the live per-launch events
    hbm_peak, bf16_peak, peak_kind = load_peaks()
    fwd_b, bwd_b, per_kernel = algorithmic_bytes(w, x)
    roof = None
    if dom and dom in live:
        cnt, ms = live[dom]
        avg_s = ms / cnt / 1000.0
        alg = per_kernel.get(dom)
        if alg is not None:
            ach = alg / avg_s / 1e9
            roof = {"bound": "hbm", "kernel": dom, "achieved": round(ach, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(ach / hbm_peak, 4), "peak_kind": peak_kind, "traffic": measured_traffic(dom, args.workload),
                    "avg_launch_us": round(avg_s * 1e6, 2), "algorithmic_bytes_per_launch": alg}
    launches = sum(c for c, _ in kern.values())
    fwd_s = statistics.mean(fwd_ms) / 1000.0
    bwd_s = statistics.mean(bwd_ms) / 1000.0
    kernel_table = {k: {"launches": c, "total_ms": round(ms, 4), "share": round(ms / max(1e-9, sum(
        m for _, m in kern.values())), 4)} for k, (c, ms) in sorted(kern.items(), key=lambda kv: -kv[1][1])}

    # ---- the other pair, for comparison (same inputs, same flush; after the timed region)
    other = None
    if world == 1:
        alt = not args.recompute
        for _ in range(3):
            flush.zero_()
            fwd(alt)
            bwd(alt)
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            ev2[i][0].record(stream)
            fwd(alt)
            bwd(alt)
            ev2[i][1].record(stream)
        torch.cuda.synchronize()
        oms = statistics.mean(a.elapsed_time(b) for a, b in ev2)
        other = {"pair": "recompute" if alt else "saved_context", "ms_per_step": round(oms, 4),
                 "value": tokens_per_step / (oms / 1000.0)}

    # ---- end-to-end through the public API with host buffers.  Every step copies its inputs from
    # pinned host memory and its outputs back.  Pipelined (the reported value): copies run on their own
    # streams into double-buffered device tensors, so step i+1's upload and step i-1's download overlap
    # step i's compute, as a data loader would; serial: everything on one stream (also reported).
    e2e = None
    if rank == 0:
        in_keys = ("q", "k", "v", "g", "beta", "dO")
        host_in = {k: x[k].cpu().pin_memory() for k in in_keys}
        outs = {"o": o, "S_T": ST, "dq": dq, "dk": dk, "dv": dv, "dg": dg, "dbeta": db}
        if dS0 is not None:
            outs["dS0"] = dS0
        host_out = {k: torch.empty_like(t, device="cpu").pin_memory() for k, t in outs.items()}
        nbuf = 2
        dev_in = [{k: torch.empty_like(x[k]) for k in in_keys} for _ in range(nbuf)]
        dev_out = [{k: torch.empty_like(t) for k, t in outs.items()} for _ in range(nbuf)]
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())
        s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()

        def compute(di, do):
            rc = fwd_call(di["q"], di["k"], di["v"], di["g"], di["beta"], do["o"], args.recompute, do["S_T"])
            assert rc == 0
            rc = bwd_call(di["q"], di["k"], di["v"], di["g"], di["beta"], di["dO"],
                          (do["dq"], do["dk"], do["dv"], do["dg"], do["dbeta"], do.get("dS0")), args.recompute)
            assert rc == 0

        def run(n, pipelined):
            hs = s_h2d if pipelined else stream
            ds = s_d2h if pipelined else stream
            ev_in = [torch.cuda.Event() for _ in range(n)]
            ev_comp = [torch.cuda.Event() for _ in range(n)]
            ev_out = [torch.cuda.Event() for _ in range(n)]
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            hs.wait_event(t0)
            for i in range(n):
                b = i % nbuf
                if pipelined and i >= nbuf:
                    hs.wait_event(ev_comp[i - nbuf])  # compute i-2 has read this input buffer
                with torch.cuda.stream(hs):
                    for k in in_keys:
                        dev_in[b][k].copy_(host_in[k], non_blocking=True)
                ev_in[i].record(hs)
                stream.wait_event(ev_in[i])
                if pipelined and i >= nbuf:
                    stream.wait_event(ev_out[i - nbuf])  # download i-2 has read this output buffer
                compute(dev_in[b], dev_out[b])
                ev_comp[i].record(stream)
                ds.wait_event(ev_comp[i])
                with torch.cuda.stream(ds):
                    for k in host_out:
                        host_out[k].copy_(dev_out[b][k], non_blocking=True)
                ev_out[i].record(ds)
            stream.wait_event(ev_out[n - 1])
            t1.record(stream)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1) / n

        n_e2e = max(3, min(args.steps, 10))
        run(2, True)
        pipe_ms = run(n_e2e, True)
        run(2, False)
        serial_ms = run(n_e2e, False)
        e2e = {"value": tokens_per_step / (pipe_ms / 1000.0), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(pipe_ms, 4), "pipelined": True,
               "serial_ms_per_step": round(serial_ms, 4),
               "serial_value": tokens_per_step / (serial_ms / 1000.0)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if x["dtype"] == "bf16" else "fp32",
            "data": "synthetic (seeded gdn_inputs; q,k raw Gaussian with in-kernel L2 norm)",
            "config": {"workload": args.workload, "B": x["q"].shape[0], "T": x["q"].shape[1], "H": H, "d": D,
                       "chunk": 64, "l2norm_in_kernel": x["l2norm"], "initial_state": x["S0"] is not None,
                       "seg_chunks": plan["seg_chunks"], "seg_first": plan["seg_first"],
                       "l2": "256 MB flush before every step, outside the events",
                       "pair": "recompute" if args.recompute else "saved_context",
                       "saved_bytes": 0 if args.recompute else saved_bytes,
                       "parallelism": f"replica x{world}"},
            "other_pair": other,
            "fwd_ms": round(1000 * fwd_s, 4), "bwd_ms": round(1000 * bwd_s, 4),
            "fwd_hbm_frac": round(fwd_b / fwd_s / 1e9 / hbm_peak, 4),
            "bwd_hbm_frac": round(bwd_b / bwd_s / 1e9 / hbm_peak, 4),
            "fwdbwd_hbm_frac": round((fwd_b + bwd_b) / (fwd_s + bwd_s) / 1e9 / hbm_peak, 4),
            "roofline": roof, "kernels": kernel_table, "gpu_launches": launches, "cpu_baseline": cpu, "e2e": e2e,
            "clocks": clk, "wall_s": round(wall, 3),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
