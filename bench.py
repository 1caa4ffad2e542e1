"""Benchmark of the compression hot path on one GB300 (one process per GPU under torchrun).

One step = qvg_quantize (T smoothing stages of Lloyd k-means + group INT2 encoding) followed
by qvg_dequantize (fused reconstruction to bf16) of every tensor of the workload, with the
inputs already resident in HBM.  Default workload: one attention layer at 1.3B-DiT shape
(12 heads x K/V = 24 tensors of 32760 tokens x 128, C=256, T=2, 10 Lloyd rounds, INT2 with
32-channel groups).

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle instead, on a
bounded sample of the same workload, and prints the same kind of line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from video_kv_cache_gb300 import synth  # noqa: E402

METRIC = "fused dequant GB/s (% HBM peak); quantize (k-means+PRQ) Mtokens/s"
DEFAULT_WORKLOAD = "layer_1p3b_32760"
L2_FLUSH_BYTES = 512 << 20


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return pk["hbm_gbs"], pk["bf16_tflops"], pk["bf16_tflops_sustained"], "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if ws > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend)
    return rank, ws


def shard(n_tensors: int, rank: int, world: int):
    """Contiguous share of the independent tensors for this rank (no data exchange)."""
    per, rem = divmod(n_tensors, world)
    lo = rank * per + min(rank, rem)
    return lo, lo + per + (1 if rank < rem else 0)


def _max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _barrier(world):
    if world > 1:
        torch.distributed.barrier()


def dequant_bytes(H, N, C, T, bits, group, out_bytes=2, n_tables=1):
    """Algorithmic bytes of one reconstruction: codes + scales + pi read, tables read once,
    output written."""
    per_tok = 128 * bits / 8 + 128 / group + T + 128 * out_bytes
    tables = T * C * 128 * 4 * n_tables
    return H * (N * per_tok + tables)


def cpu_baseline(w, steps=1, budget_s=20.0):
    """The oracle as it stands, on a bounded sample of the workload, on this host's cores."""
    import oracle
    cores = oracle.num_cores()
    X = w.make("cpu", tids=w.tids[:1])
    Xd = oracle.decode_input(X)
    # sample: whole tensors (all N tokens), as many as there are cores, capped by a quick
    # one-tensor timing so the run stays within the budget
    t0 = time.perf_counter()
    r = oracle.quantize(Xd, w.C, w.T, w.bits, w.group, w.iters, w.seed, nthreads=1)
    oracle.dequantize(r["codes"][0], r["scales"][0], r["pi"][0], r["centroids"][0], w.bits,
                      w.group)
    one = time.perf_counter() - t0
    n = int(max(1, min(w.H, cores, budget_s / max(one, 1e-3) * cores)))
    n = min(n, cores)
    Xs = w.make("cpu", tids=w.tids[:n])
    Xsd = oracle.decode_input(Xs)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        r = oracle.quantize(Xsd, w.C, w.T, w.bits, w.group, w.iters, w.seed, nthreads=cores)
        for h in range(n):
            oracle.dequantize(r["codes"][h], r["scales"][h], r["pi"][h], r["centroids"][h],
                              w.bits, w.group)
        times.append(time.perf_counter() - t0)
    dt = statistics.median(times)
    return {"value": n * w.N / dt / 1e6, "unit": "Mtokens/s", "cores": min(cores, n),
            "kind": "oracle",
            "sample": "%d of %d tensors, all %d tokens each, quantize + dequantize, %d thread(s)"
                      % (n, w.H, w.N, min(cores, n)),
            "seconds_per_step": dt}


def run_reference(args, w):
    rank, world = _dist()
    if rank != 0:
        return
    cb = None
    times = []
    for i in range(args.warmup + args.steps):
        c = cpu_baseline(w, steps=1, budget_s=args.ref_budget)
        if i >= args.warmup:
            times.append(c["seconds_per_step"])
            cb = c
    v = cb["value"]
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "Mtokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.median(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "tensors": w.H, "tokens": w.N, "C": w.C, "T": w.T,
                       "bits": w.bits, "group": w.group, "iters": w.iters},
            "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")},
            "e2e": {"value": v, "unit": "Mtokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, w):
    from video_kv_cache_gb300 import api, qvg
    from video_kv_cache_gb300 import build as qbuild
    rank, world = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    qbuild.build()
    qvg.load()
    lo, hi = shard(w.H, rank, world)
    tids = w.tids[lo:hi]
    H, N = len(tids), w.N
    X = w.make(dev, tids=tids)
    out = api.allocate(H, N, w.C, w.T, w.bits, w.group, device=dev)
    ws = api.new_workspace(H, N, w.C, w.T, dev)
    xhat = torch.empty((H, N, 128), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream()

    def quantize():
        api.quantize(X, w.C, w.T, w.bits, w.group, w.iters, w.seed, out=out, workspace=ws,
                     status=status, tensor_id_base=lo)

    def dequantize():
        api.dequantize(out, N, torch.bfloat16, out=xhat, status=status)

    for _ in range(args.warmup):
        quantize()
        dequantize()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "device status %#x" % int(status.item())

    # --- timed steps: L2 flushed before each step, each step timed with CUDA events
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    deq_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    _barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    with ClockSampler(local) as clocks:
        for k in range(args.steps):
            flush.fill_(k & 0xFF)
            ev[k][0].record(st)
            quantize()
            ev[k][1].record(st)
            dequantize()
            ev[k][2].record(st)
        # dequant alone with a cold L2, for its HBM roofline
        for k in range(args.steps):
            flush.fill_((k + 7) & 0xFF)
            deq_ev[k][0].record(st)
            dequantize()
            deq_ev[k][1].record(st)
        torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    _barrier(world)
    q_ms = [a.elapsed_time(b) for a, b, _ in ev]
    step_ms = [a.elapsed_time(c) for a, _, c in ev]
    d_ms = [a.elapsed_time(b) for a, b in deq_ev]
    step_ms_avg = _max_over_ranks(sum(step_ms) / len(step_ms), world)
    q_ms_avg = _max_over_ranks(sum(q_ms) / len(q_ms), world)
    d_ms_avg = _max_over_ranks(sum(d_ms) / len(d_ms), world)
    tokens_all = w.H * N  # whole job: every rank's tensors

    # --- end to end through the same API with host buffers (pinned), copies timed
    Xh = X.cpu().pin_memory()
    cache_h = {k: torch.empty(getattr(out, k).shape, dtype=getattr(out, k).dtype,
                              pin_memory=True) for k in ("codes", "scales", "pi", "centroids")}
    h2d = Xh.numel() * Xh.element_size()
    d2h = sum(t.numel() * t.element_size() for t in cache_h.values())
    e2e_ms = []
    for k in range(max(2, args.steps // 2)):
        flush.fill_(k & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        X.copy_(Xh, non_blocking=True)
        quantize()
        dequantize()
        for key, t in cache_h.items():
            t.copy_(getattr(out, key), non_blocking=True)
        e1.record(st)
        torch.cuda.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    e2e_avg = _max_over_ranks(sum(e2e_ms) / len(e2e_ms), world)

    hbm, tf_burst, tf_sus, src = _peaks()
    dbytes = dequant_bytes(w.H, N, w.C, w.T, w.bits, w.group) / world * world
    dq_gbs = dequant_bytes(H, N, w.C, w.T, w.bits, w.group) / (d_ms_avg * 1e-3) / 1e9
    useful_flops = 2.0 * H * N * w.C * 128 * w.iters * w.T
    n_launch_q = 1 + w.T * (4 + 3 * w.iters) + 1
    if rank == 0:
        clk = clocks.summary()
        line = {
            "metric": METRIC,
            "value": tokens_all / (step_ms_avg * 1e-3) / 1e6,
            "unit": "Mtokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_ms_avg, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "tensors": w.H, "tokens": N, "C": w.C, "T": w.T,
                       "bits": w.bits, "group": w.group, "iters": w.iters,
                       "parallelism": "dp%d (tensors sharded, no exchange)" % world,
                       "l2": "flushed (%d MiB write) before every timed step" % (L2_FLUSH_BYTES >> 20)},
            "quantize": {"ms": q_ms_avg, "mtokens_s": tokens_all / (q_ms_avg * 1e-3) / 1e6,
                         "useful_tflops": useful_flops * world / (q_ms_avg * 1e-3) / 1e12},
            "dequant": {"ms": d_ms_avg, "gbs": dq_gbs, "pct_hbm": 100.0 * dq_gbs / hbm,
                        "bytes": dbytes},
            "roofline_dequant": {"bound": "hbm", "achieved": dq_gbs, "peak": hbm, "unit": "GB/s",
                                 "frac": dq_gbs / hbm, "traffic": None, "peak_source": src},
            "e2e": {"value": tokens_all / (e2e_avg * 1e-3) / 1e6, "unit": "Mtokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms": e2e_avg},
            "gpu_launches": args.steps * (n_launch_q + 1) + args.steps,
            "wall_s_timed_region": wall,
            "clocks": clk,
        }
        if not args.no_cpu_baseline and world == 1:
            cb = cpu_baseline(w, budget_s=args.ref_budget)
            line["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=20.0)
    args = ap.parse_args()
    w = synth.workload(args.workload)
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
