"""The allocation-free entry point (mla_kv_prolog_run_noalloc) against the
handle-based one (mla_kv_prolog_run) and against the fp64 oracle, through
the C ABI.

Some callers cannot allocate device memory: an engine that plans every
byte of device memory up front, or a latency-critical path that must not
block or fail in cudaMalloc.  The no-alloc entry point serves them with a
fixed scratch array inside the library.  This file is named so that pytest
collects it last; it must pass on its own in a fresh process and after the
other tests.  Two calls in a row (different inputs and shapes) check that
the shared array's leftovers from one call do not leak into the next.  The
V2-Lite b=200 and R1 b=65 cases need two chained decode launches (128 and 64
rows per launch), which reuse the array's barrier counters within one call."""
import pytest
import torch

from mla_attention_kv_gb300 import binding as B
from mla_attention_kv_gb300 import build as BLD
from mla_attention_kv_gb300 import inputs as I

from parity import MAX_ABS, MEAN_REL, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    BLD.build()
    B.load()


def _close(name, a, b):
    a, b = a.double(), b.double()
    d = (a - b).abs()
    assert torch.isfinite(a).all(), name
    assert d.max().item() <= MAX_ABS, (name, d.max().item())
    assert d.sum().item() / max(b.abs().sum().item(), 1e-300) <= MEAN_REL, name


@pytest.mark.parametrize("cfg,b,s,seed", [(I.V2_LITE, 4, 2, 61), (I.V2_LITE, 70, 1, 62),
                                          (I.R1, 2, 1, 63), (I.V2_LITE, 200, 1, 64),
                                          (I.R1, 65, 1, 65)])
def test_noalloc_matches_handle_run_twice(oracle_mod, cfg, b, s, seed):
    for call in range(2):
        inp = I.kv_inputs(cfg, b, s, seed + 100 * call)
        d = B.to_device(inp)
        m = B.MLAProlog(cfg, b * s)
        m.set_path(B.PATH_DECODE)
        ref = m.alloc_outputs(b, s)
        m.run(b, s, d, ref)
        torch.cuda.synchronize()
        assert m.status() == 0
        m.close()
        out = {k: torch.full_like(v, float("nan")) for k, v in ref.items()}
        st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        B.mla_kv_prolog_run_noalloc(cfg, b, s, d["hidden"], d["positions"], d["W_kva"],
                                    d["gamma_kv"], d["W_kvb"], d["cos"], d["sin"],
                                    out["k_nope"], out["value"], out["k_pe"], st)
        torch.cuda.synchronize()
        assert st.item() == 0
        for k in ("k_nope", "value", "k_pe"):
            _close(k, out[k], ref[k])
        for k, r in zip(("k_nope", "value", "k_pe"), oracle_mod.kv_prolog(inp)):
            compare(k, out[k], r, oracle_mod)
