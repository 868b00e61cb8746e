"""bench.py's setup -> eager step -> e2e step flow on the CPU: the handle is
replaced by a fake that checks what each call receives (inputs and outputs
inside the staged buffers) and writes a marker into the outputs; the CUDA
device queries are stubbed and host buffers are not pinned.  The kernels,
events and graphs are the GPU tests' and the benchmark's own business; this
covers the Python plumbing around them."""
import types

import pytest
import torch

import bench
from mla_attention_kv_gb300 import binding as B

REAL = B.MLAProlog


def inside(t, buf):
    off = t.data_ptr() - buf.data_ptr()
    return 0 <= off and off + t.numel() * t.element_size() <= buf.numel() and off % 256 == 0


class FakeProlog:
    """Stands in for binding.MLAProlog: same allocation helpers, recording
    run methods."""
    alloc_outputs = REAL.alloc_outputs
    alloc_latent_outputs = REAL.alloc_latent_outputs
    alloc_paged_caches = REAL.alloc_paged_caches
    alloc_c8_outputs = REAL.alloc_c8_outputs
    made = []
    log = []  # every call of every handle, in order

    def __init__(self, cfg, max_tokens, *a, **k):
        self.cfg, self.max_tokens = cfg, max_tokens
        self.last_launches = 1
        self.calls = []
        self.packed = None
        FakeProlog.made.append(self)

    def set_path(self, path):
        self.path = path

    def close(self):
        self.closed = True

    def prepare_weights(self, d):
        self.packed = d["W_kva"].data_ptr()

    def _record(self, kind, b, s, d, out):
        assert b * s <= self.max_tokens
        self.calls.append((kind, b, s, d["hidden"], d["positions"], out))
        FakeProlog.log.append(self.calls[-1])
        for v in out.values():
            v.fill_(len(FakeProlog.log))
        return out

    def run(self, b, s, d, out, stream=None):
        return self._record("run", b, s, d, out)

    def run_latent(self, b, s, d, out, stream=None):
        return self._record("latent", b, s, d, out)

    def run_c8(self, b, s, d, scales, out, stream=None):
        assert set(scales) == {"k", "v", "kpe"}
        return self._record("c8", b, s, d, out)

    def run_paged(self, b, s, d, slots, page, out, stream=None):
        assert slots.dtype == torch.int32 and slots.numel() == b * s and page > 0
        return self._record("paged", b, s, d, out)


@pytest.fixture
def cpu_bench(monkeypatch):
    FakeProlog.made = []
    FakeProlog.log = []
    monkeypatch.setattr(B, "MLAProlog", FakeProlog)
    monkeypatch.setattr(torch.cuda, "get_device_properties",
                        lambda dev: types.SimpleNamespace(L2_cache_size=4 << 20))
    monkeypatch.setattr(torch.cuda, "synchronize", lambda dev=None: None)
    real_carve = bench.carve
    monkeypatch.setattr(bench, "carve", lambda specs, device, pin=False: real_carve(specs, device, False))
    return torch.device("cpu")


def test_decode_sweep_flow(cpu_bench):
    wl = bench.DecodeSweep()
    wl.setup(cpu_bench)
    assert wl.R >= 2 and len(FakeProlog.made) == wl.R
    assert all(m.packed is not None for m in FakeProlog.made)
    host = wl.host_inputs()
    # eager step: one call per point, on the staged views
    n = wl.step(None)
    assert n == len(wl.points)
    h2d, d2h = wl.e2e_step(None)
    assert h2d == wl.in_h.numel() and d2h == wl.out_h.numel()
    calls = FakeProlog.log
    assert len(calls) == 2 * len(wl.points)
    assert sum(len(m.calls) for m in FakeProlog.made) == len(calls)
    for (kind, b, s, hid, pos, out), (pb, ps), inp in zip(calls[len(wl.points):], wl.points, host):
        assert (kind, b, s) == ("run", pb, ps)
        assert inside(hid, wl.in_d) and inside(pos, wl.in_d)
        assert torch.equal(hid, inp["hidden"]) and torch.equal(pos, inp["positions"])
        for v in out.values():
            assert inside(v, wl.out_d)
    # the single device-to-host copy came after the calls: every output's
    # bytes in out_h carry its call's marker
    for i, (_, _, _, _, _, out) in enumerate(calls[len(wl.points):]):
        for v in out.values():
            off = v.data_ptr() - wl.out_d.data_ptr()
            back = wl.out_h[off:off + v.numel() * v.element_size()].view(v.dtype)
            assert torch.all(back == len(wl.points) + i + 1)


@pytest.mark.parametrize("name,kind", [("v2lite_tiny", "run"), ("v2lite_latent_decode", "latent"),
                                       ("v2lite_c8_decode", "c8"), ("v2lite_paged_decode", "paged"),
                                       ("w8a8_t1", "run")])
def test_single_call_flow(cpu_bench, name, kind):
    wl = bench.WORKLOADS[name]()
    wl.setup(cpu_bench)
    (m,) = FakeProlog.made
    inp = wl.host_inputs()
    h2d, d2h = wl.e2e_step(None)
    assert h2d == wl.in_h.numel() and d2h == wl.out_h.numel()
    (call,) = m.calls
    k, b, s, hid, pos, out = call
    assert (k, b, s) == (kind, wl.b, wl.s)
    assert inside(hid, wl.in_d) and inside(pos, wl.in_d)
    assert torch.equal(hid, inp["hidden"]) and torch.equal(pos, inp["positions"])
    assert out is wl.out and all(inside(v, wl.out_d) for v in out.values())
    assert torch.all(wl.out_h == wl.out_d)
    if not wl.w8:
        assert m.packed == wl.d["W_kva"].data_ptr()
