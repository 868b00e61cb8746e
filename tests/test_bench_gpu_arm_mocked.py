"""bench.py's GPU arm end to end on the CPU: run_gpu() and gpu_line() with
the handle replaced by the recording stand-in of test_bench_flow and the
CUDA runtime pieces the bench touches (streams, events, graphs, the sleep
kernel, device properties) replaced by host fakes.  What it checks is the
plumbing and the JSON contract: exactly K timed steps, the clock-triggered
re-measure, the roofline / e2e / clocks / gpu_launches keys, and a line
that serialises.  The numbers themselves are meaningless here."""
import argparse
import contextlib
import json
import time
import types

import pytest
import torch

import bench
from mla_attention_kv_gb300 import binding as B
from mla_attention_kv_gb300 import build as BLD

from test_bench_flow import FakeProlog


class FakeEvent:
    def __init__(self, enable_timing=False):
        self.t = None

    def record(self, stream=None):
        self.t = time.perf_counter()

    def elapsed_time(self, other):
        return (other.t - self.t) * 1e3


class FakeGraph:
    replays = 0

    def replay(self):
        FakeGraph.replays += 1


class FakeClocks:
    """First timed region throttled, every later one clean."""
    made = 0

    def __init__(self, index):
        FakeClocks.made += 1
        self.n = FakeClocks.made

    def stop(self):
        if self.n == 1:
            return {"sm_mhz": 1500.0, "sm_max_mhz": 2070.0, "reasons": ["hw_slowdown"], "samples": 5}
        return {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 5}


@pytest.fixture
def fake_cuda(monkeypatch):
    FakeProlog.made, FakeProlog.log = [], []
    FakeGraph.replays, FakeClocks.made = 0, 0
    monkeypatch.setattr(B, "MLAProlog", FakeProlog)
    monkeypatch.setattr(BLD, "build", lambda *a, **k: None)
    stream = types.SimpleNamespace(cuda_stream=0)
    for name, val in dict(synchronize=lambda dev=None: None, _sleep=lambda cycles: None,
                          current_stream=lambda dev=None: stream, Stream=lambda dev=None: stream,
                          Event=FakeEvent, CUDAGraph=FakeGraph,
                          stream=lambda s: contextlib.nullcontext(),
                          graph=lambda g, stream=None: contextlib.nullcontext(),
                          get_device_properties=lambda dev: types.SimpleNamespace(L2_cache_size=4 << 20)
                          ).items():
        monkeypatch.setattr(torch.cuda, name, val)
    monkeypatch.setattr(bench, "ClockSampler", FakeClocks)
    real_carve = bench.carve
    monkeypatch.setattr(bench, "carve", lambda specs, device, pin=False: real_carve(specs, device, False))
    return torch.device("cpu")


def args_for(steps=3, warmup=3):
    return argparse.Namespace(steps=steps, warmup=warmup, gpus=1, impl="gb300", no_cpu_baseline=True,
                              cpu_seconds=1.0, ref_seconds=1.0)


def check_line(line, wl, steps):
    json.dumps(line)  # serialisable as it stands
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "gpu_launches", "clocks", "e2e"):
        assert k in line, k
    assert line["steps"] == steps and line["n_gpus"] == 1 and line["higher_is_better"] is True
    assert line["config"]["workload"] == wl.describe()["workload"]
    roof = line["roofline"]
    assert roof["bound"] in ("hbm", "tensor") and roof["achieved"] > 0 and roof["peak"] > 0
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
    assert "traffic" in roof
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] == wl.in_h.numel()
    assert e2e["d2h_bytes_per_step"] == wl.out_h.numel()
    # the clean second attempt is the one reported; the first is kept beside it
    assert line["clocks_ok"] is True and line["clocks"]["reasons"] == []
    assert line["remeasured"]["why"] == "throttled: hw_slowdown"


@pytest.mark.parametrize("packed", [True, False])
def test_decode_sweep_gpu_arm(fake_cuda, packed):
    wl = bench.DecodeSweep(packed=packed)
    a = args_for(steps=3)
    r = bench.run_gpu(a, wl, 0, 1, fake_cuda)
    line = bench.gpu_line(a, wl, r, 1, "f16", False)
    check_line(line, wl, 3)
    # timed regions: graph (twice: re-measured) and eager, K steps each
    assert FakeClocks.made == 3
    assert len(r["calls"]) == 3 and all(Ts == [b * s for b, s in wl.points] for _, Ts in r["calls"])
    assert len(r["calls_eager"]) == 3 * len(wl.points)
    assert set(line["per_point"]) == {f"b{b}s{s}" for b, s in wl.points}
    assert line["gpu_launches"] == 3 * wl.graph_launches
    assert all((m.packed is not None) == packed for m in FakeProlog.made)


def test_workload_summary(fake_cuda):
    a = args_for(steps=3)
    a.workload_steps = 2
    for name in bench.EXTRA_WORKLOADS:
        out = bench.workload_summary(a, name, fake_cuda)
        json.dumps(out)
        assert out["steps"] == 2 and out["mean_call_us"] > 0 and out["tokens_per_s"] > 0
        assert out["roofline"]["frac"] == pytest.approx(out["roofline"]["achieved"] / out["roofline"]["peak"])


@pytest.mark.parametrize("name", sorted(n for n in bench.WORKLOADS if not n.startswith("decode_sweep")))
def test_single_call_gpu_arm(fake_cuda, name):
    wl = bench.WORKLOADS[name]()
    a = args_for(steps=4)
    r = bench.run_gpu(a, wl, 0, 1, fake_cuda)
    line = bench.gpu_line(a, wl, r, 1, "bf16", getattr(wl, "w8", False))
    check_line(line, wl, 4)
    assert len(r["calls"]) == 4 and all(Ts == [wl.T] for _, Ts in r["calls"])
