"""bench.py's reference arm (the CPU oracle, no GPU): the step logic runs
exactly `warmup` untimed and `steps` timed steps on samples sized to the
time budget, and `--impl reference` prints the contract's JSON line for a
single-call workload and for the decode sweep (rank 0 only)."""
import json
import os
import subprocess
import sys
import time

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class FakeWorkload:
    """Stands in for a workload: a step of size n costs `fixed` seconds plus
    `per_row` per row, and every call is recorded."""
    tokens_per_step = 200

    def __init__(self, fixed=0.02, per_row=0.001):
        self.fixed, self.per_row = fixed, per_row
        self.calls = []

    def host_inputs(self):
        return None

    def sample_rows(self, n):
        return min(n, self.tokens_per_step)

    def oracle_size(self, target, nthreads):
        return bench.fit_sample_size(self.oracle_step, self.sample_rows, self.tokens_per_step, target,
                                     nthreads)

    def oracle_step(self, k, n, nthreads):
        rows = self.sample_rows(n)
        time.sleep(self.fixed + self.per_row * rows)
        self.calls.append((k, n))
        return rows

    def sample_text(self, n):
        return f"{n} rows"


def test_oracle_steps_counts_and_sizing():
    wl = FakeWorkload()
    # 2 + 3 steps in about 1 s: 0.2 s a step -> about 180 of the 200 rows
    v, cores, text, n, el = bench.oracle_steps(wl, steps=3, warmup=2, seconds=1.0)
    calib, rest = wl.calls[:3], wl.calls[3:]
    assert [k for k, _ in calib] == [0, 1, 2] and calib[2][1] > calib[1][1]
    assert rest == [(0, n), (1, n), (2, n), (3, n), (4, n)]
    assert 120 <= n <= 200, n
    assert abs(el - 3 * (0.02 + 0.001 * n)) < 0.15
    assert abs(v - 3 * n / el) < 1e-6 * v and cores >= 1 and text == f"{n} rows"


def test_oracle_steps_whole_step_when_it_fits():
    wl = FakeWorkload(fixed=0.01, per_row=0.0001)
    _, _, _, n, _ = bench.oracle_steps(wl, steps=2, warmup=1, seconds=1.0)
    assert n == wl.tokens_per_step


def run_reference(*extra, env=None):
    e = dict(os.environ)
    e.update(env or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *extra],
                       capture_output=True, text=True, timeout=600, env=e, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]


def check_line(d, steps, warmup):
    assert d["impl"] == "reference" and d["metric"] == "tokens/s" and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["steps"] == steps and d["warmup"] == warmup
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert f"{warmup} untimed + {steps} timed steps" in cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_single_call():
    (d,) = run_reference("--workload", "v2lite_tiny", "--steps", "2", "--warmup", "3", "--ref-seconds", "2")
    check_line(d, 2, 3)
    assert d["config"]["workload"] == "v2lite_kv_prolog_tiny_b1s2"


def test_reference_arm_decode_sweep():
    (d,) = run_reference("--steps", "2", "--warmup", "3", "--ref-seconds", "1")
    check_line(d, 2, 3)
    assert d["config"]["workload"] == "v2lite_kv_prolog_decode_sweep"
    assert "calls of a V2-Lite decode sweep step per step (whole calls" in d["cpu_baseline"]["sample"]


def test_decode_sweep_samples_whole_calls(monkeypatch):
    """A sweep sample of n calls runs points k*n .. k*n + n - 1 (mod 16),
    each on all of its rows; the size is the number of mean calls that fit."""
    import oracle
    wl = bench.DecodeSweep()
    seen = []
    monkeypatch.setattr(oracle, "kv_prolog", lambda inp, rows=None, nthreads=0: seen.append((inp["b"], inp["s"], rows)))
    wl._host = [dict(b=b, s=s) for b, s in wl.points]
    assert wl.oracle_step(3, 5, 1) == sum(b * s for b, s in (wl.points * 2)[15:20])
    assert seen == [(b, s, None) for b, s in (wl.points * 2)[15:20]]
    seen.clear()
    clock = iter(range(100))
    monkeypatch.setattr(bench.time, "perf_counter", lambda: next(clock) * 0.5)  # every call 0.5 s
    assert wl.oracle_size(2.2, 1) == 4 and len(seen) == 16
    assert wl.oracle_size(100.0, 1) == 16


def test_reference_arm_other_ranks_exit_quietly():
    assert run_reference("--workload", "v2lite_tiny", env={"RANK": "1", "WORLD_SIZE": "2"}) == []
