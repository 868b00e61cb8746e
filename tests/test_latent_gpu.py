"""GPU parity of the latent-cache variant (kv_a_proj, split, RMSNorm of
compressed_kv, RoPE of k_pe; no kv_b_proj) against the fp64 oracle, through
the C ABI, on both kernels: the decode kernel (one launch per 128 / 64 rows,
raw and packed W_kva) and the tensor-core prefill kernel (with and without
the k_pe worker CTAs).  k_pe must be bit-identical to the full prolog's."""
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


def run_latent(cfg, b, s, seed, positions="decode", path=B.PATH_DECODE, rows=None,
               oracle_mod=None, packed=False, full_too=False):
    inp = I.kv_inputs(cfg, b, s, seed, positions)
    d = B.to_device(inp)
    m = B.MLAProlog(cfg, max(1, b * s))
    m.set_path(path)
    if packed:
        m.prepare_weights(d)
    out = m.alloc_latent_outputs(b, s)
    for t in out.values():
        t.fill_(float("nan"))
    m.run_latent(b, s, d, out)
    torch.cuda.synchronize()
    res = dict(inp=inp, out=out, status=m.status(), path=m.last_path, launches=m.last_launches)
    if full_too:
        full = m.alloc_outputs(b, s)
        m.run(b, s, d, full)
        torch.cuda.synchronize()
        res["full"] = full
        res["status_full"] = m.status()
    m.close()
    if oracle_mod is not None:
        lat, kpe = oracle_mod.kv_latent(inp, rows=rows)
        res["err"] = dict(latent=compare("latent", out["latent"], lat, oracle_mod),
                          k_pe=compare("k_pe", out["k_pe"], kpe, oracle_mod))
    return res


@pytest.mark.parametrize("b,s", [(1, 1), (1, 2), (17, 1), (32, 2), (128, 1), (100, 2)])
def test_latent_decode_v2lite(oracle_mod, b, s):
    r = run_latent(I.V2_LITE, b, s, 300 + b * s, oracle_mod=oracle_mod, full_too=True)
    assert r["status"] == 0 and r["path"] == B.PATH_DECODE
    assert torch.equal(r["out"]["k_pe"], r["full"]["k_pe"])


@pytest.mark.parametrize("packed", [False, True])
def test_latent_decode_r1(oracle_mod, packed):
    r = run_latent(I.R1, 64, 1, 331, oracle_mod=oracle_mod, packed=packed)
    assert r["status"] == 0 and r["path"] == B.PATH_DECODE


def test_latent_decode_small_heads(oracle_mod):
    cfg = I.small_config(I.V2_LITE, hidden=256, num_heads=1)
    r = run_latent(cfg, 3, 5, 332, oracle_mod=oracle_mod, full_too=True)
    assert r["status"] == 0
    assert torch.equal(r["out"]["k_pe"], r["full"]["k_pe"])


@pytest.mark.parametrize("T", [1024, 1000, 2048 + 37])
def test_latent_prefill_v2lite(oracle_mod, T):
    r = run_latent(I.V2_LITE, 1, T, 340 + T, positions="prefill", path=B.PATH_PREFILL,
                   oracle_mod=oracle_mod, full_too=True)
    assert r["status"] == 0 and r["path"] == B.PATH_PREFILL
    assert torch.equal(r["out"]["k_pe"], r["full"]["k_pe"])


def test_latent_prefill_r1_sampled(oracle_mod):
    b, s = 2, 8192
    rows = I.tile_rows(b, s, 512, seed=2005)
    r = run_latent(I.R1, b, s, 341, positions="prefill", path=B.PATH_PREFILL, rows=rows,
                   oracle_mod=oracle_mod)
    assert r["status"] == 0


def test_latent_decode_matches_prefill(oracle_mod):
    """Both kernels compute the same latent rows, to within the parity
    tolerance (their fp32 reduction orders differ, so a row can round to a
    neighbouring fp16 value)."""
    cfg = I.V2_LITE
    inp = I.kv_inputs(cfg, 1, 1100, 350, "prefill")
    d = B.to_device(inp)
    outs = []
    for path in (B.PATH_DECODE, B.PATH_PREFILL):
        m = B.MLAProlog(cfg, 1100)
        m.set_path(path)
        out = m.alloc_latent_outputs(1, 1100)
        m.run_latent(1, 1100, d, out)
        torch.cuda.synchronize()
        assert m.status() == 0
        m.close()
        outs.append(out)
    a, b_ = outs[0]["latent"].double(), outs[1]["latent"].double()
    d = torch.abs(a - b_)
    assert d.max().item() <= 2e-2
    assert d.sum().item() / torch.abs(a).sum().item() <= 5e-3
