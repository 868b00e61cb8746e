"""GPU parity of the tcgen05 prefill kernel against the fp64 oracle (through
the C ABI): small forced-prefill cases with ragged tiles and sequence
boundaries inside a tile, both dtypes, small head counts, the full-size
V2-Lite prefill (b=4, s=4096, T=16384) and the R1-shaped prefill (b=2,
s=8192, bf16) on sampled rows, and agreement with the decode kernel."""
import pytest
import torch

from mla_attention_kv_gb300 import binding as B
from mla_attention_kv_gb300 import build as BLD
from mla_attention_kv_gb300 import inputs as I

from parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    BLD.build()
    B.load()


def run(cfg, b, s, seed, positions, path, oracle_mod=None, rows=None):
    inp = I.kv_inputs(cfg, b, s, seed, positions)
    d = B.to_device(inp)
    m = B.MLAProlog(cfg, b * s)
    m.set_path(path)
    out = m.alloc_outputs(b, s)
    for t in out.values():
        t.fill_(float("nan"))
    m.run(b, s, d, out)
    torch.cuda.synchronize()
    st = m.status()
    res = dict(inp=inp, out=out, status=st, path=m.last_path, launches=m.last_launches)
    if oracle_mod is not None:
        ref = oracle_mod.kv_prolog(inp, rows=rows)
        res["err"] = {}
        for name, r in zip(("k_nope", "value", "k_pe"), ref):
            res["err"][name] = compare(name, out[name], r, oracle_mod)
    m.close()
    return res


@pytest.mark.parametrize("b,s", [(1, 1), (1, 100), (1, 128), (1, 129), (3, 100), (5, 61), (2, 300)])
def test_prefill_small_v2lite(oracle_mod, b, s):
    r = run(I.V2_LITE, b, s, 300 + b * s, "prefill", B.PATH_PREFILL, oracle_mod)
    assert r["status"] == 0 and r["path"] == B.PATH_PREFILL and r["launches"] == 1


@pytest.mark.parametrize("H,hidden,dtype", [(1, 64, "fp16"), (2, 128, "bf16"), (3, 192, "fp16"),
                                            (16, 2048, "bf16"), (5, 640, "bf16")])
def test_prefill_small_shapes(oracle_mod, H, hidden, dtype):
    cfg = I.small_config(I.V2_LITE, hidden=hidden, num_heads=H, dtype=dtype)
    run(cfg, 2, 150, 700 + H, "decode", B.PATH_PREFILL, oracle_mod)


def test_prefill_matches_decode_path():
    cfg = I.V2_LITE
    a = run(cfg, 2, 64, 31, "prefill", B.PATH_PREFILL)
    d = run(cfg, 2, 64, 31, "prefill", B.PATH_DECODE)
    for k in ("k_nope", "value", "k_pe"):
        diff = (a["out"][k].float() - d["out"][k].float()).abs().max().item()
        assert diff <= 2e-2, (k, diff)


def test_prefill_v2lite_full_size_sampled(oracle_mod):
    b, s = 4, 4096
    rows = I.tile_rows(b, s, 512, seed=2002)
    r = run(I.V2_LITE, b, s, I.seed_for(2), "prefill", B.PATH_AUTO, oracle_mod, rows=rows)
    assert r["status"] == 0 and r["path"] == B.PATH_PREFILL


def test_prefill_r1_full_size_sampled(oracle_mod):
    b, s = 2, 8192
    rows = I.tile_rows(b, s, 512, seed=2003)
    r = run(I.R1, b, s, I.seed_for(3), "prefill", B.PATH_AUTO, oracle_mod, rows=rows)
    assert r["status"] == 0 and r["path"] == B.PATH_PREFILL


def test_prefill_deterministic():
    a = run(I.V2_LITE, 1, 300, 5, "prefill", B.PATH_PREFILL)
    b = run(I.V2_LITE, 1, 300, 5, "prefill", B.PATH_PREFILL)
    for k in ("k_nope", "value", "k_pe"):
        assert torch.equal(a["out"][k].view(torch.int16), b["out"][k].view(torch.int16))


@pytest.mark.parametrize("cfg", [I.V2_LITE, I.R1], ids=["v2lite", "r1"])
def test_auto_path_around_threshold(oracle_mod, cfg):
    """PATH_AUTO on the dense path just below, at and just above the token
    count where it switches from the decode kernel to the prefill kernel
    (the bucketed replacement of [MIG] §源码级原理's short / long
    selection): the right kernel runs and the outputs match the oracle."""
    m = B.MLAProlog(cfg, 1)
    thr = m.auto_threshold
    m.close()
    assert thr > 1
    for T in (thr - 1, thr, thr + 1):
        rows = I.tile_rows(1, T, 64, seed=T)
        r = run(cfg, 1, T, 900 + T, "prefill", B.PATH_AUTO, oracle_mod, rows=rows)
        assert r["status"] == 0
        assert r["path"] == (B.PATH_PREFILL if T >= thr else B.PATH_DECODE), (T, thr)
