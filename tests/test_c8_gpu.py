"""GPU checks of the int8 KV-cache variant (mla_kv_prolog_run_c8) on the
decode and the prefill kernel.  Bit-exact: the codes equal the oracle's
quantiser applied to the same kernel's dtype outputs (a dense run on the
same handle), so the fused epilogue quantises exactly as specified.  Against
the fp64 oracle: codes within one step of the oracle's own codes everywhere.
The dtype values themselves may differ in the last place (the parity
tolerance allows it), which moves a code when the value sits near a
rounding boundary: with these scales (about 0.015) one bf16 unit in the last
place at |x| ~ 0.5 is about 0.13 code steps, one fp16 unit about 0.02, so the
fraction of equal codes is required to be at least 90 % (bf16) / 99 % (fp16)."""
import numpy as np
import pytest
import torch

from mla_attention_kv_gb300 import binding as B
from mla_attention_kv_gb300 import build as BLD
from mla_attention_kv_gb300 import inputs as I

pytestmark = pytest.mark.gpu
NAMES = ("k_nope", "value", "k_pe")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    BLD.build()
    B.load()


def make_scales(cfg, seed):
    """Per-channel scales near amax / 127 of the outputs' typical range."""
    g = np.random.default_rng(seed)
    H = cfg["num_heads"]
    kpe_hi = 0.04 if cfg["hidden"] <= 2048 else 0.08
    return dict(k=g.uniform(0.01, 0.02, H * 128).astype(np.float32),
                v=g.uniform(0.01, 0.02, H * 128).astype(np.float32),
                kpe=g.uniform(kpe_hi / 2, kpe_hi, 64).astype(np.float32))


def run_c8(cfg, b, s, seed, path, positions="decode", oracle_mod=None, rows=None, packed=False):
    inp = I.kv_inputs(cfg, b, s, seed, positions)
    d = B.to_device(inp)
    sc = make_scales(cfg, seed)
    scd = {k: torch.tensor(v, device="cuda") for k, v in sc.items()}
    m = B.MLAProlog(cfg, b * s)
    m.set_path(path)
    if packed:
        m.prepare_weights(d)
    q = m.alloc_c8_outputs(b, s)
    m.run_c8(b, s, d, scd, q)
    torch.cuda.synchronize()
    assert m.status() == 0
    dense = m.alloc_outputs(b, s)
    m.run(b, s, d, dense)
    torch.cuda.synchronize()
    assert m.status() == 0
    m.close()
    dt = 0 if cfg["dtype"] == "fp16" else 1
    chan = dict(k_nope=sc["k"], value=sc["v"], k_pe=sc["kpe"])
    for n in NAMES:
        g = q[n].cpu().numpy()
        x = dense[n].double().cpu().numpy()
        # scales are per channel: head-major hh*128 + e for k_nope / value
        if n == "k_pe":
            want = oracle_mod.quant_c8(x, chan[n], dt)
        else:
            H = x.shape[1]
            want = oracle_mod.quant_c8(x, chan[n].reshape(1, H, 1, 128), dt)
        assert np.array_equal(g, want), n
    if oracle_mod is not None:
        ref = oracle_mod.kv_prolog(inp, rows=rows)
        for n, r in zip(NAMES, ref):
            g = q[n].cpu().numpy()
            m_ = ~np.isnan(r)
            if n == "k_pe":
                o = oracle_mod.quant_c8(r, chan[n], dt)
            else:
                o = oracle_mod.quant_c8(r, chan[n].reshape(1, r.shape[1], 1, 128), dt)
            diff = np.abs(g.astype(np.int32) - o.astype(np.int32))[m_]
            assert diff.max() <= 1, n
            assert (diff == 0).mean() >= (0.99 if dt == 0 else 0.90), (n, (diff == 0).mean())


@pytest.mark.parametrize("b,s", [(1, 2), (64, 1), (100, 2)])
def test_c8_decode_v2lite(oracle_mod, b, s):
    run_c8(I.V2_LITE, b, s, 500 + b * s, B.PATH_DECODE, oracle_mod=oracle_mod)


@pytest.mark.parametrize("packed", [False, True])
def test_c8_decode_r1(oracle_mod, packed):
    # packed R1 weights: kv_b on the tensor cores, the same int8 store epilogue
    run_c8(I.R1, 64, 1, 510, B.PATH_DECODE, oracle_mod=oracle_mod, packed=packed)


@pytest.mark.parametrize("T", [1024, 1061])
def test_c8_prefill_v2lite(oracle_mod, T):
    rows = I.tile_rows(1, T, 512, seed=T + 1)
    run_c8(I.V2_LITE, 1, T, 520 + T, B.PATH_PREFILL, positions="prefill", oracle_mod=oracle_mod,
           rows=rows)
