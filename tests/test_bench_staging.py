"""bench.py's host/device staging (no GPU: staged on the CPU, unpinned):
carve() lays tensors out back to back at 256-byte boundaries, and each
workload's stage_io() puts every input row and every output in one buffer
whose views the calls use, so that one copy of the buffer moves all of them
(the e2e step's single host-to-device and device-to-host copies)."""
import types

import pytest
import torch

import bench
from mla_attention_kv_gb300 import binding as B


def test_carve_alignment_and_aliasing():
    specs = [((3,), torch.int32), ((2, 5), torch.float16), ((1,), torch.int8), ((4, 4), torch.bfloat16)]
    buf, views = bench.carve(specs, "cpu")
    base = buf.data_ptr()
    ends = []
    for v, (shape, dt) in zip(views, specs):
        assert tuple(v.shape) == shape and v.dtype == dt and v.is_contiguous()
        off = v.data_ptr() - base
        assert off % 256 == 0
        ends.append((off, off + v.numel() * v.element_size()))
    for (a0, a1), (b0, b1) in zip(ends, ends[1:]):
        assert a1 <= b0  # in order, disjoint
    assert ends[-1][1] <= buf.numel()
    # writes through a view land in the buffer
    views[1].fill_(1.5)
    assert torch.equal(buf[256:256 + 20].view(torch.float16), torch.full((10,), 1.5, dtype=torch.float16))


def test_carve_dicts_keeps_keys_and_shapes():
    meta = [dict(a=torch.empty(2, 3, device="meta"), b=torch.empty(7, dtype=torch.int32, device="meta")),
            dict(c=torch.empty(1, 1, 5, dtype=torch.float16, device="meta"))]
    buf, ds = bench.carve_dicts(meta, "cpu")
    assert [list(d) for d in ds] == [["a", "b"], ["c"]]
    for m, d in zip(meta, ds):
        for k in m:
            assert d[k].shape == m[k].shape and d[k].dtype == m[k].dtype and d[k].device.type == "cpu"


def outs_meta(cfg, kind, b, s, paged=None):
    fake = types.SimpleNamespace(cfg=cfg)
    if kind == "latent":
        return B.MLAProlog.alloc_latent_outputs(fake, b, s, "meta")
    if kind == "c8":
        return B.MLAProlog.alloc_c8_outputs(fake, b, s, "meta")
    if kind == "paged":
        return B.MLAProlog.alloc_paged_caches(fake, paged[1], paged[0], "meta")
    return B.MLAProlog.alloc_outputs(fake, b, s, "meta")


def check_one_copy_moves_outputs(out_d, out_h, outs):
    # fill every output view with its own value, copy the buffer once, and
    # read each output back through the same layout on the host side
    for i, d in enumerate(outs):
        for j, v in enumerate(d.values()):
            v.fill_(i * 8 + j + 1)
    out_h.copy_(out_d)
    buf = out_h
    for i, d in enumerate(outs):
        for j, v in enumerate(d.values()):
            off = v.data_ptr() - out_d.data_ptr()
            back = buf[off:off + v.numel() * v.element_size()].view(v.dtype)
            assert torch.all(back == i * 8 + j + 1)


def test_decode_sweep_staging():
    wl = bench.DecodeSweep()
    outs = [outs_meta(wl.cfg, "dense", b, s) for b, s in wl.points]
    wl.stage_io("cpu", outs, pin=False)
    host = wl.host_inputs()
    assert len(wl.pt) == len(wl.points) == 16
    seen = []
    for (b, s), p, inp in zip(wl.points, wl.pt, host):
        assert (p["b"], p["s"]) == (b, s)
        for k in ("hidden", "positions"):
            v = p[k]
            assert torch.equal(v, inp[k]) and v.dtype == inp[k].dtype
            off = v.data_ptr() - wl.in_d.data_ptr()
            assert off % 256 == 0 and 0 <= off and off + v.numel() * v.element_size() <= wl.in_d.numel()
            seen.append((off, off + v.numel() * v.element_size()))
    seen.sort()
    assert all(a[1] <= b[0] for a, b in zip(seen, seen[1:]))
    # the host twin has the same layout and contents: one copy reproduces in_d
    assert wl.in_h.shape == wl.in_d.shape and torch.equal(wl.in_h, wl.in_d)
    assert wl.in_h.numel() >= sum(b * s * (2 * 2048 + 4) for b, s in wl.points)
    for o, m in zip(wl.out, outs):
        for k in m:
            assert o[k].shape == m[k].shape and o[k].dtype == m[k].dtype
            assert (o[k].data_ptr() - wl.out_d.data_ptr()) % 256 == 0
    assert wl.out_h.shape == wl.out_d.shape
    check_one_copy_moves_outputs(wl.out_d, wl.out_h, wl.out)


@pytest.mark.parametrize("name,kind", [("v2lite_tiny", "dense"), ("v2lite_latent_decode", "latent"),
                                       ("v2lite_c8_decode", "c8"), ("v2lite_paged_decode", "paged"),
                                       ("w8a8_t1", "dense")])
def test_single_call_staging(name, kind):
    wl = bench.WORKLOADS[name]()
    inp = wl.host_inputs()
    wl.d = {k: v for k, v in inp.items()}
    out = outs_meta(wl.cfg, kind, wl.b, wl.s, wl.paged)
    wl.stage_io("cpu", out, pin=False)
    for k in ("hidden", "positions"):
        v = wl.d[k]
        assert torch.equal(v, inp[k])
        off = v.data_ptr() - wl.in_d.data_ptr()
        assert off % 256 == 0 and off + v.numel() * v.element_size() <= wl.in_d.numel()
    # the weights are untouched
    assert wl.d["W_kva"] is inp["W_kva"]
    assert torch.equal(wl.in_h, wl.in_d)
    assert list(wl.out) == list(out)
    check_one_copy_moves_outputs(wl.out_d, wl.out_h, [wl.out])
