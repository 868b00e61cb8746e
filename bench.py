"""Benchmark of the GB300 MLA KV prolog.

Default workload: the DeepSeek-V2-Lite decode sweep (s in {1, 2} x b in
{1, 2, 4, ..., 128}; fp16; 765 token rows per step).  One step runs the whole
prolog once per sweep point through the C ABI.  Metric: tokens/s (whole job,
all ranks), plus the fraction of the HBM roofline of the decode kernel.

Timing rules kept here:
  * W untimed warm-up steps, then exactly K timed steps between CUDA events
    on the launching stream, with a barrier + synchronize on both sides; the
    max over ranks is reported.
  * The weights are re-read from HBM every call: the step cycles through
    enough copies of the weights (same values) to exceed twice the L2
    capacity, as consecutive layers of a model would.
  * Launches are enqueued ahead of the GPU (a device-side sleep before the
    start event), so the timed region measures the device, and one CUDA
    event between consecutive launches gives each launch's duration.
  * e2e: the same steps through the public binding with pinned host inputs
    copied in and the three outputs copied back every step (wall clock).

``--impl reference`` times the CPU oracle (the plain fp64 definition of
the prolog) on a bounded sample of the same workload; there is no other
reference implementation of this path.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mla_attention_kv_gb300 import inputs as I  # noqa: E402

SWEEP_B = [1, 2, 4, 8, 16, 32, 64, 128]
SWEEP_S = [1, 2]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------ workload
class DecodeSweep:
    name = "v2lite_kv_prolog_decode_sweep"

    def __init__(self):
        self.cfg = I.V2_LITE
        self.points = [(b, s) for s in SWEEP_S for b in SWEEP_B]
        self.tokens_per_step = sum(b * s for b, s in self.points)

    def describe(self):
        return {"workload": self.name, "model": "DeepSeek-V2-Lite KV prolog", "hidden": 2048,
                "kv_lora_rank": 512, "rope_dim": 64, "num_heads": 16, "nope_dim": 128,
                "v_dim": 128, "points": [f"b{b}s{s}" for b, s in self.points],
                "tokens_per_step": self.tokens_per_step, "positions": "uniform per sequence in [0,4095]"}

    def weight_bytes(self):
        c = self.cfg
        return 2 * (c["hidden"] * 576 + 512 + 512 * c["num_heads"] * 256)

    def alg_bytes(self, T):
        # weights once + per token: hidden row, position, cos+sin rows, outputs
        c = self.cfg
        per_tok = 2 * c["hidden"] + 4 + 2 * 64 * 4 + 2 * (c["num_heads"] * 256 + 64)
        return self.weight_bytes() + per_tok * T

    def setup(self, dev):
        from mla_attention_kv_gb300 import binding as B
        self.B = B
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.R = max(2, math.ceil(2 * l2 / self.weight_bytes()))
        base = I.kv_inputs(self.cfg, 1, 1, I.seed_for(1, 0))
        self.wcopies = []
        for _ in range(self.R):
            self.wcopies.append({k: base[k].to(dev) for k in ("W_kva", "gamma_kv", "W_kvb")})
        self.cos = base["cos"].to(dev)
        self.sin = base["sin"].to(dev)
        self.pt = []
        for i, (b, s) in enumerate(self.points):
            inp = I.kv_inputs(self.cfg, b, s, I.seed_for(1, i))
            self.pt.append(dict(b=b, s=s, hidden=inp["hidden"].to(dev),
                                positions=inp["positions"].to(dev),
                                hidden_h=inp["hidden"].pin_memory(),
                                positions_h=inp["positions"].pin_memory()))
        self.m = B.MLAProlog(self.cfg, max(b * s for b, s in self.points))
        self.out = [self.m.alloc_outputs(p["b"], p["s"], dev) for p in self.pt]
        self.out_h = [{k: torch.empty_like(v, device="cpu").pin_memory() for k, v in o.items()}
                      for o in self.out]
        self.calls = 0

    def _run(self, i, stream):
        p = self.pt[i]
        w = self.wcopies[self.calls % self.R]
        self.calls += 1
        d = dict(hidden=p["hidden"], positions=p["positions"], cos=self.cos, sin=self.sin, **w)
        self.m.run(p["b"], p["s"], d, self.out[i], stream)
        return self.m.last_launches

    def step(self, stream, events=None):
        """One pass over the sweep; with `events`, record one event after
        each launch (events[0] must be recorded by the caller before)."""
        n = 0
        for i in range(len(self.pt)):
            n += self._run(i, stream)
            if events is not None:
                events.append(torch.cuda.Event(enable_timing=True))
                events[-1].record(stream)
        return n

    def step_bytes(self):
        return [self.alg_bytes(b * s) for b, s in self.points]

    def e2e_step(self, stream):
        h2d = d2h = 0
        for i, p in enumerate(self.pt):
            p["hidden"].copy_(p["hidden_h"], non_blocking=True)
            p["positions"].copy_(p["positions_h"], non_blocking=True)
            h2d += p["hidden_h"].numel() * 2 + p["positions_h"].numel() * 4
            self._run(i, stream)
            for k, v in self.out[i].items():
                self.out_h[i][k].copy_(v, non_blocking=True)
                d2h += v.numel() * v.element_size()
        return h2d, d2h

    # CPU oracle on a bounded sample
    def cpu_sample(self, seconds):
        import oracle
        oracle.build()
        nt = os.cpu_count() or 1
        done = 0
        t0 = time.perf_counter()
        pts = 0
        while True:
            i = pts % len(self.points)
            b, s = self.points[i]
            inp = I.kv_inputs(self.cfg, b, s, I.seed_for(1, i))
            oracle.kv_prolog(inp, nthreads=nt)
            done += b * s
            pts += 1
            if time.perf_counter() - t0 >= seconds:
                break
        el = time.perf_counter() - t0
        return done / el, min(nt, oracle.max_threads()), \
            f"{pts} sweep points in order ({done} token rows) of the V2-Lite decode sweep, fp64 oracle, {el:.1f} s"


WORKLOADS = {"decode_sweep": DecodeSweep}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.p = None
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "100", "-i",
                                       str(index)], stdout=subprocess.PIPE,
                                      stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.p.terminate()
        out, _ = self.p.communicate(timeout=10)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ------------------------------------------------------------------ main
def run_gpu(args, wl, rank, world, dev):
    from mla_attention_kv_gb300 import build as BLD
    if rank == 0:
        BLD.build()
    if world > 1:
        torch.distributed.barrier()
    BLD.build()
    wl.setup(dev)
    stream = torch.cuda.current_stream(dev)

    # warm-up (also measures host enqueue time per step)
    t0 = time.perf_counter()
    for _ in range(args.warmup):
        launches_per_step = wl.step(stream)
    torch.cuda.synchronize(dev)
    host_per_step = (time.perf_counter() - t0) / max(1, args.warmup)

    # timed region
    events = []
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    sleep_s = min(5.0, 1.5 * host_per_step * args.steps + 0.05)
    torch.cuda._sleep(int(sleep_s * 2.0e9))
    start = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    events.append(start)
    total_launches = 0
    for _ in range(args.steps):
        total_launches += wl.step(stream, events)
    end = events[-1]
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ms = start.elapsed_time(end)
    durs = [events[i].elapsed_time(events[i + 1]) for i in range(len(events) - 1)]
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    if durs[-1] <= 0:
        log("warning: zero-duration events")

    # e2e through the public binding with host buffers
    for _ in range(2):
        wl.e2e_step(stream)
    torch.cuda.synchronize(dev)
    e2e_steps = max(3, args.steps // 4)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        h2d, d2h = wl.e2e_step(stream)
    torch.cuda.synchronize(dev)
    e2e_s = time.perf_counter() - t0
    if world > 1:
        t = torch.tensor([e2e_s], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_s = float(t.item())
    return dict(ms=ms, durs=durs, clk=clk, launches=total_launches,
                launches_per_step=launches_per_step, e2e_s=e2e_s, e2e_steps=e2e_steps,
                h2d=h2d, d2h=d2h, host_per_step=host_per_step)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="decode_sweep", choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    wl = WORKLOADS[args.workload]()

    if args.impl == "reference":
        if rank != 0:
            return
        per_step_s = None
        # each step: the oracle over a bounded sample of the workload
        v, cores, sample = wl.cpu_sample(min(args.cpu_seconds, 20.0))
        line = {"metric": "tokens/s", "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": None,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic", "impl": "reference",
                "config": dict(wl.describe(), parallelism="none (host cores)"),
                "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores,
                                 "kind": "oracle", "sample": sample},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        if per_step_s:
            line["ms_per_step"] = per_step_s * 1e3
        print(json.dumps(line), flush=True)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    r = run_gpu(args, wl, rank, world, dev)

    tokens = wl.tokens_per_step * args.steps * world
    value = tokens / (r["ms"] / 1e3)
    peaks, peak_kind = measured_peaks()
    step_bytes = wl.step_bytes()
    n_launch = len(r["durs"])
    # algorithmic bytes of each timed launch, aligned with the events
    per_call = []
    for _ in range(args.steps):
        per_call.extend(step_bytes)
    alg = sum(per_call)
    dur_s = sum(r["durs"]) / 1e3
    achieved = alg / dur_s / 1e9
    line = {
        "metric": "tokens/s", "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms"] / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded N(0,1) hidden, N(0,0.02) weights, gamma 1+N(0,0.1))",
        "config": dict(wl.describe(), parallelism=f"replicas x{world}" if world > 1 else "none",
                       l2="weights rotated over %d copies (> 2x L2) so every call reads them from HBM" % wl.R),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                     "peak_kind": peak_kind, "kernel": "decode_kernel",
                     "launches_timed": n_launch,
                     "mean_launch_us": 1e3 * sum(r["durs"]) / n_launch},
        "gpu_launches": r["launches"],
        "clocks": r["clk"],
        "e2e": {"value": wl.tokens_per_step * r["e2e_steps"] * world / r["e2e_s"], "unit": "tokens/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
    }
    # per-point detail: mean launch time and roofline fraction of each sweep point
    npts = len(wl.points)
    detail = {}
    for j, (b, s) in enumerate(wl.points):
        ds = [r["durs"][k] for k in range(j, n_launch, npts)]
        us = 1e3 * statistics.mean(ds)
        detail[f"b{b}s{s}"] = {"T": b * s, "us": round(us, 3),
                               "tokens_per_s": b * s / (us * 1e-6),
                               "hbm_frac": wl.alg_bytes(b * s) / (us * 1e-6) / 1e9 / peaks["hbm_gbs"]}
    line["per_point"] = detail
    if rank == 0 and not args.no_cpu_baseline:
        v, cores, sample = wl.cpu_sample(args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
