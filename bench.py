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
    copied in and the outputs copied back every step (wall clock); for the
    decode sweep the copies run on streams of their own, issued through the
    CUDA driver API, and overlap the neighbouring steps' calls.
  * nvidia-smi clocks are sampled during the timed region; a region that saw
    a hardware or thermal slowdown, or SM clocks well below the maximum with
    no reason, is measured once more and the first attempt is reported
    beside the second ("remeasured").

``--impl reference`` times the CPU oracle (the plain fp64 definition of
the prolog) on the host cores: W untimed and K timed steps, each the whole
workload step or a bounded sample of it (``oracle_steps``); there is no
other reference implementation of this path.
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


# ------------------------------------------------------------------ copies
class DriverCopies:
    """Host<->device copies, event records and stream waits of the e2e steps
    through the CUDA driver API (ctypes on libcuda): a few microseconds of
    host time each, where torch's pinned-memory copy takes about 12 us to
    issue, which made the e2e loop host-bound.  `ok` is False where the
    driver library cannot be loaded (the e2e step then uses torch)."""

    def __init__(self):
        import ctypes
        self.ok = False
        try:
            L = ctypes.CDLL("libcuda.so.1")
        except OSError:
            return
        P, Z = ctypes.c_void_p, ctypes.c_size_t
        self.h2d, self.d2h = L.cuMemcpyHtoDAsync_v2, L.cuMemcpyDtoHAsync_v2
        self.h2d.argtypes = [ctypes.c_uint64, P, Z, P]
        self.d2h.argtypes = [P, ctypes.c_uint64, Z, P]
        self.record, self.wait = L.cuEventRecord, L.cuStreamWaitEvent
        self.record.argtypes = [P, P]
        self.wait.argtypes = [P, P, ctypes.c_uint]
        for f in (self.h2d, self.d2h, self.record, self.wait):
            f.restype = ctypes.c_int
        self.ok = True

    @staticmethod
    def check(code, what):
        if code != 0:
            raise RuntimeError(f"{what} failed: CUresult {code}")


# ------------------------------------------------------------------ workload
def carve(specs, device, pin=False):
    """One buffer holding tensors of the (shape, dtype) `specs` back to back,
    each at a 256-byte boundary (the C ABI wants 16-byte aligned pointers),
    so that a step's inputs or outputs cross between host and device in one
    copy.  Returns (buffer, views); pin=True puts the buffer in page-locked
    host memory."""
    offs, total = [], 0
    for shape, dt in specs:
        n = math.prod(shape) * torch.empty((), dtype=dt).element_size()
        offs.append((total, n))
        total += -(-n // 256) * 256
    buf = torch.empty(max(total, 256), dtype=torch.uint8, device=device, pin_memory=pin)
    views = [buf[o:o + n].view(dt).view(shape) for (o, n), (shape, dt) in zip(offs, specs)]
    return buf, views


def carve_dicts(dicts, device, pin=False):
    """carve() for a list of dicts of tensors (any device, "meta" included):
    returns (buffer, list of dicts of views with the same keys, shapes and
    dtypes)."""
    buf, views = carve([(tuple(v.shape), v.dtype) for d in dicts for v in d.values()], device, pin)
    it = iter(views)
    return buf, [{k: next(it) for k in d} for d in dicts]


class DecodeSweep:
    """The V2-Lite decode sweep.  packed: every weight copy gets the decode
    kernel's packed snapshot (mla_kv_prolog_prepare_weights, once, outside
    the timed region); otherwise the calls read the raw [in, out] weights."""

    def __init__(self, packed=True):
        self.packed = packed
        self.name = "v2lite_kv_prolog_decode_sweep" + ("" if packed else "_raw_weights")
        self.cfg = I.V2_LITE
        self.points = [(b, s) for s in SWEEP_S for b in SWEEP_B]
        self.tokens_per_step = sum(b * s for b, s in self.points)

    def describe(self):
        return {"workload": self.name, "model": "DeepSeek-V2-Lite KV prolog", "hidden": 2048,
                "kv_lora_rank": 512, "rope_dim": 64, "num_heads": 16, "nope_dim": 128,
                "v_dim": 128, "points": [f"b{b}s{s}" for b, s in self.points],
                "tokens_per_step": self.tokens_per_step, "positions": "uniform per sequence in [0,4095]",
                "weights": ("one handle per weight copy, packed once by mla_kv_prolog_prepare_weights "
                            "outside the timed region" if self.packed else
                            "raw [in, out] weights passed to every call (no packed snapshot)")}

    def weight_bytes(self):
        c = self.cfg
        return 2 * (c["hidden"] * 576 + 512 + 512 * c["num_heads"] * 256)

    def flops(self, T):
        c = self.cfg
        return 2.0 * T * (c["hidden"] * 576 + 512 * c["num_heads"] * 256)

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
        # one handle per weight copy, each with its packed snapshot (a serving
        # engine packs every layer's weights once at load time)
        tmax = max(b * s for b, s in self.points)
        self.ms = []
        for w in self.wcopies:
            m = B.MLAProlog(self.cfg, tmax)
            if self.packed:
                m.prepare_weights(w)
            self.ms.append(m)
        torch.cuda.synchronize(dev)
        self.m = self.ms[0]
        self.stage_io(dev, [self.m.alloc_outputs(b, s, "meta") for b, s in self.points])
        torch.cuda.synchronize(dev)
        self.calls = 0

    def stage_io(self, dev, outs, pin=True):
        """Every point's hidden rows and positions in one device buffer
        `in_d`, every point's outputs (shapes of the dicts `outs`) in one
        device buffer `out_d`, each with a host twin (`in_h`, `out_h`) of the
        same layout; the calls use views into the device buffers, so that an
        e2e step moves its inputs and outputs in one copy each."""
        ins = [{"hidden": inp["hidden"], "positions": inp["positions"]} for inp in self.host_inputs()]
        self.in_h, views_h = carve_dicts(ins, "cpu", pin)
        self.in_d, views_d = carve_dicts(ins, dev)
        for src, dst in zip(ins, views_h):
            for k in src:
                dst[k].copy_(src[k])
        self.in_d.copy_(self.in_h)
        self.pt = [dict(b=b, s=s, **v) for (b, s), v in zip(self.points, views_d)]
        self.out_d, self.out = carve_dicts(outs, dev)
        self.out_h, _ = carve_dicts(outs, "cpu", pin)
        # a second device set for the e2e steps (double buffering, below)
        self.e2e_sets = None
        if self.in_d.is_cuda:
            in_d2, views_d2 = carve_dicts(ins, dev)
            out_d2, out2 = carve_dicts(outs, dev)
            pt2 = [dict(b=b, s=s, **v) for (b, s), v in zip(self.points, views_d2)]
            self.e2e_sets = [(self.in_d, self.out_d, self.pt, self.out), (in_d2, out_d2, pt2, out2)]
            self.e2e_k = 0

    def _run(self, i, stream, pt=None, out=None):
        p = (pt or self.pt)[i]
        w = self.wcopies[self.calls % self.R]
        m = self.ms[self.calls % self.R]
        self.calls += 1
        d = dict(hidden=p["hidden"], positions=p["positions"], cos=self.cos, sin=self.sin, **w)
        m.run(p["b"], p["s"], d, (out or self.out)[i], stream)
        self.cl_calls = getattr(self, "cl_calls", 0) + getattr(m, "last_cluster_launches", 0)
        return m.last_launches

    def step(self, stream, events=None, intervals=None):
        """One pass over the sweep; with `events`, record one event after
        each call (events[-1] is the event before the first call) and the
        index pair of each call's interval in `intervals`."""
        n = 0
        for i in range(len(self.pt)):
            n += self._run(i, stream)
            if events is not None:
                events.append(torch.cuda.Event(enable_timing=True))
                events[-1].record(stream)
                intervals.append((len(events) - 2, len(events) - 1, [self.pt[i]["b"] * self.pt[i]["s"]]))
        return n

    def step_bytes(self):
        return [self.alg_bytes(b * s) for b, s in self.points]

    def capture(self, dev):
        """One CUDA graph per rotation offset: graph p holds the 16 calls of a
        step that starts at weight copy 16p (mod R)."""
        st = torch.cuda.Stream(dev)
        graphs = []
        saved = self.calls
        for gi in range(self.R):
            self.calls = (gi * len(self.pt)) % self.R
            g = torch.cuda.CUDAGraph()
            n = 0
            with torch.cuda.stream(st):
                with torch.cuda.graph(g, stream=st):
                    for i in range(len(self.pt)):
                        n += self._run(i, st)
            graphs.append(g)
            self.graph_launches = n
        self.calls = saved
        torch.cuda.synchronize(dev)
        return graphs

    def graph_step(self, k, graphs, stream, events, intervals):
        events.append(torch.cuda.Event(enable_timing=True))
        events[-1].record(stream)
        graphs[k % len(graphs)].replay()
        events.append(torch.cuda.Event(enable_timing=True))
        events[-1].record(stream)
        intervals.append((len(events) - 2, len(events) - 1, [b * s for b, s in self.points]))
        return self.graph_launches

    def e2e_step(self, stream):
        """One step from host buffers: every point's inputs in one
        host-to-device copy, the 16 calls, every output in one device-to-host
        copy (pinned host memory; bytes are the copied buffers').  On a GPU the
        two copies run on streams of their own and the steps alternate between
        two device buffer sets, so that a step's copies overlap the calls of
        its neighbours (as a serving loop would stage the next batch while
        this one runs); every step still makes both copies of its own."""
        if self.e2e_sets is None or stream is None:
            self.in_d.copy_(self.in_h, non_blocking=True)
            for i in range(len(self.pt)):
                self._run(i, stream)
            self.out_h.copy_(self.out_d, non_blocking=True)
            return self.in_h.numel(), self.out_h.numel()
        if getattr(self, "e2e_streams", None) is None:
            self.e2e_streams = (torch.cuda.Stream(), torch.cuda.Stream())
            self.e2e_calls_done = [None, None]  # per set: the event after its last calls
            self.e2e_out_read = [None, None]    # per set: the event after its last D2H copy
            self.cu = DriverCopies()
            if self.cu.ok:
                # per set: staged, calls done, outputs read (recorded again every use)
                self.e2e_ev = [[torch.cuda.Event() for _ in range(3)] for _ in range(2)]
                self.e2e_used = [False, False]
                for evs in self.e2e_ev:  # create the driver events now
                    for e in evs:
                        e.record(self.e2e_streams[0])
                torch.cuda.synchronize()
        up, down = self.e2e_streams
        if self.cu.ok:
            return self._e2e_step_driver(stream, up, down)
        k = self.e2e_k % 2
        self.e2e_k += 1
        in_d, out_d, pt, out = self.e2e_sets[k]
        # inputs: the set's previous calls must have read it
        if self.e2e_calls_done[k] is not None:
            up.wait_event(self.e2e_calls_done[k])
        with torch.cuda.stream(up):
            in_d.copy_(self.in_h, non_blocking=True)
        staged = torch.cuda.Event()
        staged.record(up)
        # the calls: after the inputs landed and the set's previous outputs were read
        stream.wait_event(staged)
        if self.e2e_out_read[k] is not None:
            stream.wait_event(self.e2e_out_read[k])
        for i in range(len(pt)):
            self._run(i, stream, pt, out)
        done = torch.cuda.Event()
        done.record(stream)
        self.e2e_calls_done[k] = done
        # outputs
        down.wait_event(done)
        with torch.cuda.stream(down):
            self.out_h.copy_(out_d, non_blocking=True)
        read = torch.cuda.Event()
        read.record(down)
        self.e2e_out_read[k] = read
        return self.in_h.numel(), self.out_h.numel()

    def _e2e_step_driver(self, stream, up, down):
        """e2e_step with the copies, records and waits issued through the
        driver API (same order and dependencies)."""
        cu = self.cu
        k = self.e2e_k % 2
        self.e2e_k += 1
        in_d, out_d, pt, out = self.e2e_sets[k]
        staged, done, read = (e.cuda_event for e in self.e2e_ev[k])
        s_up, s_down, s_run = up.cuda_stream, down.cuda_stream, stream.cuda_stream
        if self.e2e_used[k]:  # the set's previous calls must have read its inputs
            cu.check(cu.wait(s_up, done, 0), "cuStreamWaitEvent")
        cu.check(cu.h2d(in_d.data_ptr(), self.in_h.data_ptr(), self.in_h.numel(), s_up), "cuMemcpyHtoDAsync")
        cu.check(cu.record(staged, s_up), "cuEventRecord")
        cu.check(cu.wait(s_run, staged, 0), "cuStreamWaitEvent")
        if self.e2e_used[k]:  # and its previous outputs must have been read
            cu.check(cu.wait(s_run, read, 0), "cuStreamWaitEvent")
        for i in range(len(pt)):
            self._run(i, stream, pt, out)
        cu.check(cu.record(done, s_run), "cuEventRecord")
        cu.check(cu.wait(s_down, done, 0), "cuStreamWaitEvent")
        cu.check(cu.d2h(self.out_h.data_ptr(), out_d.data_ptr(), self.out_h.numel(), s_down), "cuMemcpyDtoHAsync")
        cu.check(cu.record(read, s_down), "cuEventRecord")
        self.e2e_used[k] = True
        return self.in_h.numel(), self.out_h.numel()

    def host_inputs(self):
        """The seeded host inputs of every sweep point (built once)."""
        if getattr(self, "_host", None) is None:
            self._host = [I.kv_inputs(self.cfg, b, s, I.seed_for(1, i)) for i, (b, s) in enumerate(self.points)]
        return self._host

    # CPU oracle on a bounded sample: n whole calls of the sweep per step
    # (consecutive points, cyclic), so that every call keeps the workload's
    # own ratio of rows to the oracle's fixed cost per call
    def oracle_size(self, target, nthreads):
        """Points per step: one untimed pass over the sweep times each
        point's call; the largest n whose mean step (n calls) fits target."""
        import oracle
        taus = []
        for inp in self.host_inputs():
            t0 = time.perf_counter()
            oracle.kv_prolog(inp, nthreads=nthreads)
            taus.append(time.perf_counter() - t0)
        mean = sum(taus) / len(taus)
        return int(max(1, min(len(self.points), target // max(mean, 1e-9))))

    def oracle_step(self, k, n, nthreads):
        """Oracle on the k-th bounded sample of the sweep: sweep points
        k*n .. k*n + n - 1 (mod 16), each a whole call.  Returns the rows."""
        import oracle
        done = 0
        host = self.host_inputs()
        for j in range(n):
            i = (k * n + j) % len(self.points)
            oracle.kv_prolog(host[i], nthreads=nthreads)
            done += self.points[i][0] * self.points[i][1]
        return done

    def sample_text(self, n):
        return (f"{n} of the 16 calls of a V2-Lite decode sweep step per step (whole calls, "
                f"consecutive points, cyclic), fp64 oracle")


class SingleCall:
    """One prolog call per step on one configuration (prefill, R1, W8A8, or
    the latent-cache variant: kv_a_proj + RMSNorm + RoPE(k_pe), no kv_b_proj)."""

    def __init__(self, name, cfg, b, s, positions, path, seed, latent=False, paged=None, c8=False):
        self.name, self.cfg, self.b, self.s = name, cfg, b, s
        self.positions, self.path, self.seed = positions, path, seed
        self.T = b * s
        self.points = [(b, s)]
        self.tokens_per_step = self.T
        self.w8 = cfg.get("quant") == "w8a8"
        self.latent = latent
        self.paged = paged  # (page_size, num_blocks): outputs scattered into a paged KV cache
        self.c8 = c8        # int8 KV-cache outputs with per-channel scales

    def describe(self):
        c = self.cfg
        d = {"workload": self.name, "model": c["name"], "hidden": c["hidden"], "num_heads": c["num_heads"],
             "b": self.b, "s": self.s, "T": self.T, "dtype": c["dtype"], "positions": self.positions}
        if self.w8:
            d["q_lora_rank"] = c["q_lora_rank"]
            d["quant"] = "w8a8 (int8 weights, per-token int8 activations, int32 accumulators)"
        if self.latent:
            d["variant"] = "latent cache: normalised compressed_kv [T, 512] + k_pe, no kv_b_proj"
        if self.c8:
            d["variant"] = "int8 KV cache: k_nope / value / k_pe codes with per-channel fp32 scales"
        if self.paged:
            d["variant"] = ("paged KV cache of %d blocks of %d rows: a random block table, each sequence's "
                            "rows at consecutive offsets of its blocks (decode: offset = position %% %d)"
                            % (self.paged[1], self.paged[0], self.paged[0]))
        return d

    def weight_bytes(self):
        c = self.cfg
        h, H, r = c["hidden"], c["num_heads"], 512
        if self.w8:
            rq = c["q_lora_rank"]
            return (h * (rq + 576) + rq * H * 192 + r * H * 256) + 4 * (rq + 576 + H * 192 + H * 256) + 2 * (rq + r)
        if self.latent:
            return 2 * (h * 576 + r)
        return 2 * (h * 576 + r + r * H * 256)

    def flops(self, T):
        c = self.cfg
        h, H = c["hidden"], c["num_heads"]
        if self.w8:
            rq = c["q_lora_rank"]
            return 2.0 * T * (h * (rq + 576) + rq * H * 192 + 512 * H * 256)
        if self.latent:
            return 2.0 * T * h * 576
        return 2.0 * T * (h * 576 + 512 * H * 256)

    def alg_bytes(self, T):
        c = self.cfg
        H = c["num_heads"]
        out = 2 * (512 + 64) if self.latent else 2 * (H * 256 + 64) + (2 * H * 192 if self.w8 else 0)
        if self.c8:
            out = H * 256 + 64 + 4 * (H * 256 + 64) / max(T, 1)  # int8 codes; the scales once per call
        return self.weight_bytes() + T * (2 * c["hidden"] + 4 + 2 * 64 * 4 + out)

    def host_inputs(self):
        """The seeded host inputs of the call (built once)."""
        if getattr(self, "host", None) is None:
            gen = I.w8a8_inputs if self.w8 else I.kv_inputs
            self.host = gen(self.cfg, self.b, self.s, self.seed, self.positions)
        return self.host

    def setup(self, dev):
        from mla_attention_kv_gb300 import binding as B
        self.B = B
        inp = self.host_inputs()
        self.d = B.to_device(inp, dev)
        self.R = 1
        self.m = B.MLAProlog(self.cfg, self.T)
        if not self.w8:
            self.m.set_path(self.path)
            self.m.prepare_weights(self.d)  # packed snapshot for the decode path
            torch.cuda.synchronize(dev)
        if self.paged:
            # a block table as a serving engine keeps it: random physical
            # blocks, a sequence's rows at consecutive offsets within them
            page, nblk = self.paged
            nbps = (self.s + page - 1) // page
            g = torch.Generator().manual_seed(self.seed)
            table = torch.randperm(nblk, generator=g)[:self.b * nbps].view(self.b, nbps)
            t = torch.arange(self.T)
            bi, si = t // self.s, t % self.s
            if self.s == 1:
                off = inp["positions"].long() % page
                slot = table[bi, 0] * page + off
            else:
                slot = table[bi, si // page] * page + si % page
            self.slots = slot.to(torch.int32).to(dev)
            out = self.m.alloc_paged_caches(nblk, page, "meta")
        elif self.latent:
            out = self.m.alloc_latent_outputs(self.b, self.s, "meta")
        elif self.c8:
            g = torch.Generator().manual_seed(self.seed)
            H = self.cfg["num_heads"]
            hi = 0.04 if self.cfg["hidden"] <= 2048 else 0.08
            self.scales = dict(k=(0.01 + 0.01 * torch.rand(H * 128, generator=g)).to(dev),
                               v=(0.01 + 0.01 * torch.rand(H * 128, generator=g)).to(dev),
                               kpe=(hi / 2 + hi / 2 * torch.rand(64, generator=g)).to(dev))
            out = self.m.alloc_c8_outputs(self.b, self.s, "meta")
        else:
            out = self.m.alloc_outputs(self.b, self.s, "meta")
        self.stage_io(dev, out)
        torch.cuda.synchronize(dev)
        # L2 flush between timed calls when the inputs fit in L2: a 2x L2 buffer
        # is written, then another 2x L2 buffer is read, so that none of the
        # call's data is in L2 and no dirty line is left to be written back
        # during the call
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.flush = None
        if self.alg_bytes(self.T) < 2 * l2:
            self.flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
            self.flush_rd = torch.ones(2 * l2 // 4, dtype=torch.float32, device=dev)
            self.flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def stage_io(self, dev, out, pin=True):
        """The hidden rows and positions in one device buffer `in_d` (the
        call's `d` points into it), the outputs (shapes of the dict `out`) in
        one device buffer `out_d`, each with a host twin (`in_h`, `out_h`)
        of the same layout, so that an e2e step moves its inputs and outputs
        in one copy each."""
        inp = self.host_inputs()
        ins = [{"hidden": inp["hidden"], "positions": inp["positions"]}]
        self.in_h, (vh,) = carve_dicts(ins, "cpu", pin)
        self.in_d, (vd,) = carve_dicts(ins, dev)
        for k in vh:
            vh[k].copy_(ins[0][k])
        self.in_d.copy_(self.in_h)
        self.d["hidden"], self.d["positions"] = vd["hidden"], vd["positions"]
        self.out_d, (self.out,) = carve_dicts([out], dev)
        self.out_h, _ = carve_dicts([out], "cpu", pin)

    def call(self, stream):
        if self.paged:
            self.m.run_paged(self.b, self.s, self.d, self.slots, self.paged[0], self.out, stream)
        elif self.latent:
            self.m.run_latent(self.b, self.s, self.d, self.out, stream)
        elif self.c8:
            self.m.run_c8(self.b, self.s, self.d, self.scales, self.out, stream)
        else:
            self.m.run(self.b, self.s, self.d, self.out, stream)
        self.cl_calls = getattr(self, "cl_calls", 0) + getattr(self.m, "last_cluster_launches", 0)

    def flush_l2(self):
        self.flush.zero_()
        torch.sum(self.flush_rd, dim=0, out=self.flush_sink)

    def step(self, stream, events=None, intervals=None):
        if self.flush is not None and events is not None:
            self.flush_l2()
            events.append(torch.cuda.Event(enable_timing=True))
            events[-1].record(stream)
        self.call(stream)
        if events is not None:
            events.append(torch.cuda.Event(enable_timing=True))
            events[-1].record(stream)
            intervals.append((len(events) - 2, len(events) - 1, [self.T]))
        return self.m.last_launches

    def step_bytes(self):
        return [self.alg_bytes(self.T)]

    def capture(self, dev):
        st = torch.cuda.Stream(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(st):
            with torch.cuda.graph(g, stream=st):
                self.call(st)
        self.graph_launches = self.m.last_launches
        torch.cuda.synchronize(dev)
        return [g]

    def graph_step(self, k, graphs, stream, events, intervals):
        if self.flush is not None:
            self.flush_l2()
        events.append(torch.cuda.Event(enable_timing=True))
        events[-1].record(stream)
        graphs[0].replay()
        events.append(torch.cuda.Event(enable_timing=True))
        events[-1].record(stream)
        intervals.append((len(events) - 2, len(events) - 1, [self.T]))
        return self.graph_launches

    def e2e_step(self, stream):
        """One call from host buffers: the inputs in one host-to-device copy,
        the outputs in one device-to-host copy (pinned host memory)."""
        self.in_d.copy_(self.in_h, non_blocking=True)
        self.call(stream)
        self.out_h.copy_(self.out_d, non_blocking=True)
        return self.in_h.numel(), self.out_h.numel()

    def oracle_size(self, target, nthreads):
        """Rows per step: the largest sample whose predicted time fits target."""
        return fit_sample_size(self.oracle_step, lambda n: min(n, self.T), self.T, target, nthreads)

    def oracle_step(self, k, n, nthreads):
        """Oracle on the k-th bounded sample of the call: token rows
        k*n .. k*n + n - 1 (mod T) in one oracle call.  Returns the rows."""
        import oracle
        fn = oracle.w8a8_prolog if self.w8 else (oracle.kv_latent if self.latent else oracle.kv_prolog)
        rows = sorted({(k * n + i) % self.T for i in range(n)})
        fn(self.host_inputs(), rows=rows, nthreads=nthreads)
        return len(rows)

    def sample_text(self, n):
        return (f"{n} token rows of {self.name} per step (consecutive, cyclic), fp64 oracle, "
                f"per-call weight promotion included")


def _single(name, cfg, b, s, positions, path_name, seed, latent=False, paged=None, c8=False):
    return lambda: SingleCall(name, cfg, b, s, positions, {"decode": 1, "prefill": 2, "auto": 0}[path_name],
                              seed, latent, paged, c8)


WORKLOADS = {
    "decode_sweep": DecodeSweep,
    "decode_sweep_raw": lambda: DecodeSweep(packed=False),
    "v2lite_tiny": _single("v2lite_kv_prolog_tiny_b1s2", I.V2_LITE, 1, 2, [7, 8], "auto", 1000),
    "v2lite_prefill": _single("v2lite_kv_prolog_prefill_b4s4096", I.V2_LITE, 4, 4096, "prefill", "auto", 1002),
    "r1_decode": _single("r1_kv_prolog_decode_b64s1", I.R1, 64, 1, "decode", "auto", 1003),
    "r1_prefill": _single("r1_kv_prolog_prefill_b2s8192", I.R1, 2, 8192, "prefill", "auto", 1003),
    "w8a8_t1": _single("r1_w8a8_prolog_T1", I.R1_W8A8, 1, 1, "decode", "auto", 1004),
    "w8a8_t64": _single("r1_w8a8_prolog_T64", I.R1_W8A8, 64, 1, "decode", "auto", 1004),
    "w8a8_t8192": _single("r1_w8a8_prolog_T8192", I.R1_W8A8, 1, 8192, "prefill", "auto", 1004),
    "v2lite_latent_decode": _single("v2lite_kv_latent_decode_b64s1", I.V2_LITE, 64, 1, "decode", "auto",
                                    1005, latent=True),
    "r1_latent_prefill": _single("r1_kv_latent_prefill_b2s8192", I.R1, 2, 8192, "prefill", "auto", 1005,
                                 latent=True),
    "v2lite_paged_decode": _single("v2lite_kv_prolog_paged_decode_b64s1", I.V2_LITE, 64, 1, "decode", "auto",
                                   1006, paged=(16, 64)),
    "r1_paged_prefill": _single("r1_kv_prolog_paged_prefill_b2s8192", I.R1, 2, 8192, "prefill", "auto", 1006,
                                paged=(64, 288)),
    "v2lite_c8_decode": _single("v2lite_kv_prolog_c8_decode_b64s1", I.V2_LITE, 64, 1, "decode", "auto", 1007,
                                c8=True),
    "r1_c8_prefill": _single("r1_kv_prolog_c8_prefill_b2s8192", I.R1, 2, 8192, "prefill", "auto", 1007, c8=True),
}


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


def fit_sample_size(run, rows, top, target, nthreads):
    """The largest sample size n <= top whose predicted time fits `target`
    seconds, for a sample made of one oracle call on rows(n) token rows
    (`run(k, n, nthreads)` runs the k-th such sample).  One untimed call
    first (the oracle's first touch of its buffers), then two calls at sizes
    n1 and about 16 n1 separate the call's fixed cost (weight promotion)
    from its cost per row."""
    def timed(k, n):
        t0 = time.perf_counter()
        run(k, n, nthreads)
        return time.perf_counter() - t0

    n1 = 1
    while n1 < top and rows(n1) < max(nthreads, 8):
        n1 *= 2
    n1 = min(n1, top)
    n2 = min(top, 16 * n1)
    r1, r2 = rows(n1), rows(n2)
    timed(0, n1)
    t1 = timed(1, n1)
    t2 = timed(2, n2) if r2 > r1 else t1
    per_row = (t2 - t1) / (r2 - r1) if r2 > r1 and t2 > t1 else t2 / r2
    fixed = max(0.0, t1 - per_row * r1)
    lo, hi = 1, top
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if fixed + per_row * rows(mid) <= target:
            lo = mid
        else:
            hi = mid - 1
    return lo


def oracle_steps(wl, steps, warmup, seconds):
    """Time the CPU oracle on the host cores: `warmup` untimed steps, then
    exactly `steps` timed steps, each a bounded sample of the workload
    (`wl.oracle_step(k, n)`; the workload's `oracle_size` picks n from an
    untimed calibration so that all warmup + steps take about `seconds`).
    Returns (tokens/s, threads used, description of the sample, size
    parameter, timed seconds)."""
    import oracle
    oracle.build()
    nt = os.cpu_count() or 1
    wl.host_inputs()
    steps = max(1, steps)
    n = wl.oracle_size(seconds / (steps + warmup), nt)
    for k in range(warmup):
        wl.oracle_step(k, n, nt)
    done = 0
    t0 = time.perf_counter()
    for k in range(steps):
        done += wl.oracle_step(warmup + k, n, nt)
    el = time.perf_counter() - t0
    return done / el, min(nt, oracle.max_threads()), wl.sample_text(n), n, el


def clocks_rejected(clk):
    """Why a timed region's clock record makes its number unacceptable, or
    None: a hardware or thermal slowdown seen at any sample, or a median SM
    clock well below the maximum with no reason given (a leftover clock
    lock).  A power cap alone is normal under load and is kept."""
    reasons = set(clk.get("reasons") or [])
    bad = reasons & {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    if bad:
        return "throttled: " + ", ".join(sorted(bad))
    sm, smax = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    if sm and smax and sm < 0.85 * smax and "sw_power_cap" not in reasons:
        return f"median SM clock {sm:.0f} of {smax:.0f} MHz with no reason"
    return None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ------------------------------------------------------------------ main
def max_over_ranks(x: float, world: int, device) -> float:
    """The largest value of x over the ranks: the job's time is its slowest
    rank's (every rank runs the same replicated work)."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_step: int, steps: int, world: int, ms: float) -> float:
    """Whole-job throughput of N independent replicas (weak scaling): the
    tokens all ranks processed over the slowest rank's time."""
    return tokens_per_step * steps * world / (ms / 1e3)


# Workloads measured beside the default decode sweep (one GPU): every other
# configuration of the benchmark, each as its own graph-replayed timed region.
EXTRA_WORKLOADS = ["decode_sweep_raw", "v2lite_tiny", "v2lite_prefill", "r1_decode", "r1_prefill",
                   "w8a8_t1", "w8a8_t64", "w8a8_t8192"]


def run_gpu(args, wl, rank, world, dev, full=True):
    """Time wl: W warm-up steps, then K graph-replayed steps (re-measured
    once if the clocks disqualify them); with full, also the same K steps
    launched eagerly and the e2e pass from host buffers."""
    from mla_attention_kv_gb300 import build as BLD
    if rank == 0:
        BLD.build()
    if world > 1:
        torch.distributed.barrier()
    BLD.build()
    wl.setup(dev)
    stream = torch.cuda.current_stream(dev)

    # warm-up (also measures the host enqueue time of a step)
    t0 = time.perf_counter()
    for _ in range(args.warmup):
        wl.step(stream)
    torch.cuda.synchronize(dev)
    host_per_step = (time.perf_counter() - t0) / max(1, args.warmup)

    # CUDA graphs of the steps (how a serving engine issues repeated decode
    # steps): captured once, replayed in the timed region
    graphs = wl.capture(dev)
    for _ in range(2):  # upload and warm every graph before the timed region
        for g in graphs:
            g.replay()
    torch.cuda.synchronize(dev)

    def timed(run_step):
        events, intervals = [], []
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        clocks = ClockSampler(dev.index if dev.index is not None else 0)
        sleep_s = min(5.0, 1.5 * host_per_step * args.steps + 0.05)
        torch.cuda._sleep(int(sleep_s * 2.0e9))
        start = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        events.append(start)
        launches = 0
        for k in range(args.steps):
            launches += run_step(k, events, intervals)
        end = events[-1]
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        clk = clocks.stop()
        region_ms = start.elapsed_time(end)
        calls = [(events[a].elapsed_time(events[b]), Ts) for a, b, Ts in intervals]
        # with an L2 flush between calls, the flush is not part of the work
        ms = sum(c for c, _ in calls) if getattr(wl, "flush", None) is not None else region_ms
        ms = max_over_ranks(ms, world, dev)
        return ms, region_ms, calls, clk, launches

    # timed region: exactly K steps (graph replays) between CUDA events on the launching stream
    def graph_run(k, ev, iv):
        return wl.graph_step(k, graphs, stream, ev, iv)

    ms, region_ms, calls, clk, total_launches = timed(graph_run)
    # a region whose clocks disqualify it is measured once more (every rank
    # takes the same decision), and the first attempt is reported beside it
    first = None
    why = clocks_rejected(clk)
    if max_over_ranks(1.0 if why else 0.0, world, dev) > 0:
        first = {"ms_per_step": ms / args.steps, "clocks": clk, "why": why or "another rank's clocks"}
        ms, region_ms, calls, clk, total_launches = timed(graph_run)
    if not full:
        return dict(ms=ms, region_ms=region_ms, calls=calls, clk=clk, launches=total_launches,
                    host_per_step=host_per_step, first_attempt=first)
    # the same K steps launched eagerly through the binding, call by call
    ms_e, _, calls_e, clk_e, _ = timed(lambda k, ev, iv: wl.step(stream, ev, iv))

    # e2e through the public binding with host buffers
    for _ in range(2):
        wl.e2e_step(stream)
    torch.cuda.synchronize(dev)
    # as many steps as the timed region (at least 8), so that filling and
    # draining the copy pipeline (one step's copies) weighs little
    e2e_steps = max(8, args.steps)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        h2d, d2h = wl.e2e_step(stream)
    torch.cuda.synchronize(dev)
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, world, dev)
    return dict(ms=ms, region_ms=region_ms, calls=calls, clk=clk, launches=total_launches,
                e2e_s=e2e_s, e2e_steps=e2e_steps, h2d=h2d, d2h=d2h, host_per_step=host_per_step,
                ms_eager=ms_e, calls_eager=calls_e, clk_eager=clk_e, first_attempt=first)


def kernel_traffic(kernel: str, T: int, model: str = ""):
    """DRAM bytes of one call of `kernel` at T rows (entry "<model>:<T>") from
    the committed ncu summary, or None when the summary is missing
    or was taken on a different version of the kernel's sources (the sha256
    of their concatenation no longer matches)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        srcs = t[kernel]["source"]
        h = hashlib.sha256()
        for src in ([srcs] if isinstance(srcs, str) else srcs):
            h.update(open(os.path.join(ROOT, "mla_attention_kv_gb300", "csrc", src), "rb").read())
        if h.hexdigest()[:16] != t[kernel]["sha256_16"]:
            return None
        return t[kernel]["bytes_per_call"].get("%s:%d" % (model, T))
    except Exception:
        return None


def roofline(wl, calls, is_w8):
    """Roofline of the timed calls [(ms, [T, ...]), ...]: algorithmic bytes
    or FLOPs (whichever takes longer at the measured peak) over the calls'
    summed CUDA-event time, against that peak; plus the committed ncu DRAM
    traffic per call when it matches the kernel source."""
    peaks, peak_kind = measured_peaks()
    Tlist = [T for _, Ts in calls for T in Ts]
    alg_bytes = sum(wl.alg_bytes(T) for T in Tlist)
    alg_flops = sum(wl.flops(T) for T in Tlist)
    call_s = sum(c for c, _ in calls) / 1e3
    # the bound is the resource whose time at peak is larger; the W8A8 int8
    # products run as exact bf16 tensor-core products, so their peak is bf16's
    bw = peaks["hbm_gbs"] * 1e9
    tensor_peak = peaks["bf16_tflops"] * 1e12
    tensor_unit = "TFLOP/s (bf16 tensor peak; int8 products as exact bf16)" if is_w8 else "TFLOP/s"
    t_mem, t_cmp = alg_bytes / bw, alg_flops / tensor_peak
    m = getattr(wl, "m", None)
    last = getattr(m, "last_path", 1) if m is not None else 1
    path = "prefill" if (not is_w8 and last == 2) else "decode"
    kernel = {"prefill": "prefill_kernel", "decode": "decode_kernel"}[path] if not is_w8 else "w8a8 pipeline"
    if getattr(wl, "latent", False):
        kernel += " (latent variant)"
    if getattr(wl, "paged", None):
        kernel += " (paged cache)"
    if getattr(wl, "c8", False):
        kernel += " (int8 cache)"
    # launches of at most 16 rows on the packed V2-Lite snapshot run the
    # cluster decode kernel (its traffic is under the same entry)
    label = kernel + (" + decode_cl_kernel (launches of <= 16 rows)" if getattr(wl, "cl_calls", 0) else "")
    if t_mem >= t_cmp:
        achieved = alg_bytes / call_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"]}
    else:
        achieved = alg_flops / call_s / 1e12
        peak = tensor_peak / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": tensor_unit,
                "frac": achieved / peak}
    Ts = sorted(set(Tlist))
    model = wl.cfg["name"]
    tr = [kernel_traffic(kernel, T, model) for T in Ts]
    roof["traffic"] = None if any(x is None for x in tr) else \
        sum(kernel_traffic(kernel, T, model) for T in Tlist) / len(Tlist)
    roof.update({"peak_kind": peak_kind, "kernel": label, "calls_timed": len(Tlist),
                 "mean_call_us": 1e6 * call_s / len(Tlist),
                 "algorithmic_bytes_per_call": alg_bytes / len(Tlist),
                 "algorithmic_flops_per_call": alg_flops / len(Tlist),
                 "timing": "CUDA events around each CUDA-graph replay of a step"})
    return roof


def workload_summary(args, name, dev):
    """One other workload, timed like the headline (graph replays, L2 rule,
    clocks) with args.workload_steps steps: per-call time, tokens/s,
    roofline and clocks."""
    wl = WORKLOADS[name]()
    a = argparse.Namespace(**vars(args))
    a.steps, a.warmup = args.workload_steps, 3
    r = run_gpu(a, wl, 0, 1, dev, full=False)
    calls = r["calls"]
    ntok = sum(T for _, Ts in calls for T in Ts)
    out = {"config": wl.describe(), "steps": a.steps, "ms_per_step": r["ms"] / a.steps,
           "mean_call_us": 1e3 * sum(c for c, _ in calls) / sum(len(Ts) for _, Ts in calls),
           "tokens_per_s": ntok / (sum(c for c, _ in calls) / 1e3),
           "roofline": roofline(wl, calls, getattr(wl, "w8", False)),
           "gpu_launches": r["launches"], "clocks": r["clk"], "clocks_ok": clocks_rejected(r["clk"]) is None}
    if r["first_attempt"] is not None:
        out["remeasured"] = r["first_attempt"]
    for m in getattr(wl, "ms", [getattr(wl, "m", None)]):
        if m is not None:
            m.close()
    del wl
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return out


def gpu_line(args, wl, r, world, dtype, is_w8):
    """The JSON line of the GPU arm from run_gpu's measurements: whole-job
    tokens/s, the roofline of the dominant kernel, clocks, e2e, the eager
    pass and (for the sweep) per-point figures; cpu_baseline is added by
    the caller."""
    value = job_tokens_per_s(wl.tokens_per_step, args.steps, world, r["ms"])
    peaks, _ = measured_peaks()
    roof = roofline(wl, r["calls"], is_w8)
    line = {
        "metric": "tokens/s", "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms"] / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
        "data": "synthetic (seeded N(0,1) hidden, N(0,0.02) weights, gamma 1+N(0,0.1))",
        "config": dict(wl.describe(), parallelism=f"replicas x{world}" if world > 1 else "none",
                       l2=("weights rotated over %d copies (> 2x L2) so every call reads them from HBM" % wl.R
                           if getattr(wl, "flush", None) is None else
                           "L2 flushed between timed calls (a 2x L2 buffer written, then another 2x L2 "
                           "buffer read: none of the call's data in L2, no dirty lines); flush time excluded")),
        "roofline": roof,
        "gpu_launches": r["launches"],
        "clocks": r["clk"],
        "clocks_ok": clocks_rejected(r["clk"]) is None,
        "e2e": {"value": job_tokens_per_s(wl.tokens_per_step, r["e2e_steps"], world, r["e2e_s"] * 1e3),
                "unit": "tokens/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
    }
    if r["first_attempt"] is not None:
        line["remeasured"] = r["first_attempt"]
    ce = r["calls_eager"]
    line["eager"] = {"value": job_tokens_per_s(wl.tokens_per_step, args.steps, world, r["ms_eager"]), "ms_per_step": r["ms_eager"] / args.steps,
                     "mean_call_us": 1e3 * sum(c for c, _ in ce) / len(ce), "clocks": r["clk_eager"],
                     "note": "the same steps launched call by call through the binding (no CUDA graph)"}
    if len(wl.points) > 1:
        npts = len(wl.points)
        detail = {}
        for j, (b, s_) in enumerate(wl.points):
            ds = [ce[k][0] for k in range(j, len(ce), npts)]
            us = 1e3 * statistics.mean(ds)
            detail[f"b{b}s{s_}"] = {"T": b * s_, "us": round(us, 3), "tokens_per_s": b * s_ / (us * 1e-6),
                                    "hbm_frac": wl.alg_bytes(b * s_) / (us * 1e-6) / 1e9 / peaks["hbm_gbs"]}
        line["per_point"] = detail
        line["per_point_timing"] = "CUDA events around each call of the eager pass"
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="decode_sweep", choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="seconds of the oracle's steps in the cpu_baseline leg")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="seconds of the oracle's warm-up + timed steps under --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload-steps", type=int, default=10,
                    help="timed steps of each other workload measured beside the default sweep")
    ap.add_argument("--no-workloads", action="store_true",
                    help="measure only the chosen workload (no 'workloads' object)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    wl = WORKLOADS[args.workload]()
    is_w8 = getattr(wl, "w8", False)
    dtype = "int8/int32 (bf16 io)" if is_w8 else ("f16" if wl.cfg["dtype"] == "fp16" else "bf16")

    if args.impl == "reference":
        if rank != 0:
            return
        v, cores, sample, n, el = oracle_steps(wl, args.steps, args.warmup, args.ref_seconds)
        sample += f"; {args.warmup} untimed + {args.steps} timed steps, {el:.1f} s timed"
        line = {"metric": "tokens/s", "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": wl.tokens_per_step / v * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "impl": "reference",
                "config": dict(wl.describe(), parallelism="none (host cores)"),
                "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores,
                                 "kind": "oracle", "sample": sample},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    r = run_gpu(args, wl, rank, world, dev)

    line = gpu_line(args, wl, r, world, dtype, is_w8)
    if args.workload == "decode_sweep" and world == 1 and not args.no_workloads:
        line["workloads"] = {}
        for name in EXTRA_WORKLOADS:
            try:
                line["workloads"][name] = workload_summary(args, name, dev)
            except Exception as e:  # a failure is reported in the line, not hidden
                line["workloads"][name] = {"error": repr(e)[:300]}
    if rank == 0 and not args.no_cpu_baseline:
        v, cores, sample, n, el = oracle_steps(wl, 4, 1, args.cpu_seconds)
        sample += f"; 1 untimed + 4 timed steps, {el:.1f} s timed"
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
