"""GPU parity of the fused decode kernel against the fp64 oracle (through the
C ABI).  Covers the tiny V2-Lite case (b=1, s=2, positions {7, 8}), the
single-token shape of the pages' golden case (b=1, s=1), every point of the
V2-Lite decode sweep (s in {1, 2} x b in {1 .. 128}), the R1-shaped decode
(b=64, s=1, bf16), ragged token counts around the 16-row m-tiles and the
64-row launch chunks, small head counts, determinism, the position check
and the bounded device wait."""
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


def run_case(cfg, b, s, seed, positions="decode", path=B.PATH_DECODE, max_tokens=None,
             rows=None, oracle_mod=None, nan_fill=True, packed=False):
    inp = I.kv_inputs(cfg, b, s, seed, positions)
    d = B.to_device(inp)
    m = B.MLAProlog(cfg, max_tokens or max(1, b * s))
    m.set_path(path)
    if packed:
        m.prepare_weights(d)
    out = m.alloc_outputs(b, s)
    if nan_fill:
        for t in out.values():
            t.fill_(float("nan"))
    m.run(b, s, d, out)
    torch.cuda.synchronize()
    st = m.status()
    res = dict(inp=inp, out=out, status=st, launches=m.last_launches, path=m.last_path)
    if oracle_mod is not None:
        ref = oracle_mod.kv_prolog(inp, rows=rows)
        res["err"] = {}
        for name, r in zip(("k_nope", "value", "k_pe"), ref):
            res["err"][name] = compare(name, out[name], r, oracle_mod)
    m.close()
    return res


def test_tiny_config_v2lite(oracle_mod):
    r = run_case(I.V2_LITE, 1, 2, I.seed_for(0), positions=[7, 8], oracle_mod=oracle_mod)
    assert r["status"] == 0 and r["launches"] == 1


def test_single_token_golden_shape(oracle_mod):
    # shapes of the pages' golden case: hidden [1,1,2048] -> [1,16,1,128] x2, [1,1,1,64]
    r = run_case(I.V2_LITE, 1, 1, 7, oracle_mod=oracle_mod)
    assert tuple(r["out"]["k_nope"].shape) == (1, 16, 1, 128)
    assert tuple(r["out"]["k_pe"].shape) == (1, 1, 1, 64)


@pytest.mark.parametrize("s", [1, 2])
@pytest.mark.parametrize("b", [1, 2, 4, 8, 16, 32, 64, 128])
def test_decode_sweep_v2lite(oracle_mod, b, s):
    point = [1, 2, 4, 8, 16, 32, 64, 128].index(b) + 8 * (s - 1)
    r = run_case(I.V2_LITE, b, s, I.seed_for(1, point), oracle_mod=oracle_mod)
    assert r["status"] == 0


def test_r1_decode(oracle_mod):
    r = run_case(I.R1, 64, 1, I.seed_for(3), oracle_mod=oracle_mod)
    assert r["status"] == 0


def rows_per_launch(cfg):
    """Token rows one decode launch takes: 128 when the CTA's whole W_kvb
    slice stays resident in shared memory (V2-Lite on a GPU with at least
    128 SMs), else 64."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return 128 if (cfg["num_heads"] <= 16 and sms >= 128) else 64


@pytest.mark.parametrize("T", [3, 15, 17, 63, 64, 65, 127, 128, 129, 200, 256, 257])
def test_ragged_token_counts(oracle_mod, T):
    r = run_case(I.V2_LITE, T, 1, 500 + T, oracle_mod=oracle_mod)
    tt = rows_per_launch(I.V2_LITE)
    assert r["status"] == 0 and r["launches"] == (T + tt - 1) // tt


def test_r1_ragged_two_launches(oracle_mod):
    r = run_case(I.R1, 65, 1, I.seed_for(3, 65), oracle_mod=oracle_mod)
    assert r["status"] == 0 and r["launches"] == 2


@pytest.mark.parametrize("H,hidden,dtype", [(1, 64, "fp16"), (3, 192, "bf16"), (5, 640, "fp16"),
                                            (16, 2048, "bf16")])
def test_small_shapes(oracle_mod, H, hidden, dtype):
    cfg = I.small_config(I.V2_LITE, hidden=hidden, num_heads=H, dtype=dtype)
    run_case(cfg, 3, 2, 900 + H, oracle_mod=oracle_mod)


def test_deterministic():
    a = run_case(I.V2_LITE, 8, 2, 42)
    b = run_case(I.V2_LITE, 8, 2, 42)
    for k in ("k_nope", "value", "k_pe"):
        assert torch.equal(a["out"][k].view(torch.int16), b["out"][k].view(torch.int16))


def test_bad_position_is_flagged_and_clamped(oracle_mod):
    cfg = I.V2_LITE
    pos = [5, 4096, -3, 100]  # rows 1 and 2 are out of range
    r = run_case(cfg, 4, 1, 77, positions=pos)
    assert r["status"] == 7
    # rows with valid positions are still exact; k_nope/value never depend on position
    ref = oracle_mod.kv_prolog(dict(r["inp"], positions=torch.tensor([5, 0, 0, 100], dtype=torch.int32)),
                               rows=[0, 3])
    compare("k_pe", r["out"]["k_pe"][[0, 3]], ref[2][[0, 3]], oracle_mod)
    ref_all = oracle_mod.kv_prolog(dict(r["inp"], positions=torch.tensor([5, 0, 0, 100], dtype=torch.int32)))
    compare("k_nope", r["out"]["k_nope"], ref_all[0], oracle_mod)


def test_device_wait_budget_expires_cleanly():
    """A 1 ns wait budget makes the grid barrier give up: the kernel must
    return (no hang), report MLA_ERR_DEVICE_TIMEOUT, and the next run on a
    normal handle must be correct again."""
    cfg = I.V2_LITE
    inp = I.kv_inputs(cfg, 2, 1, 3)
    d = B.to_device(inp)
    m = B.MLAProlog(cfg, 2, spin_budget_ns=1)
    m.set_path(B.PATH_DECODE)
    out = m.alloc_outputs(2, 1)
    m.run(2, 1, d, out)
    torch.cuda.synchronize()
    assert m.status() == 6
    assert m.status() == 0  # cleared
    m.close()
    run_case(cfg, 2, 1, 3)


def test_host_errors_on_device_buffers():
    cfg = I.V2_LITE
    inp = I.kv_inputs(cfg, 1, 2, 1)
    d = B.to_device(inp)
    m = B.MLAProlog(cfg, 2)
    out = m.alloc_outputs(1, 2)
    with pytest.raises(B.MLAError) as e:
        m.run(2, 2, d, out)  # 4 tokens > max_tokens 2
    assert e.value.code == 3
    raw = torch.empty(d["hidden"].numel() + 8, dtype=torch.float16, device="cuda")
    mis = raw[1:1 + d["hidden"].numel()].view_as(d["hidden"])
    with pytest.raises(B.MLAError) as e:
        m.run(1, 2, dict(d, hidden=mis), out)
    assert e.value.code == 4
    m.run(0, 2, d, out)  # T = 0 is a no-op
    assert m.last_launches == 0
    m.close()


# ---------------------------------------------------------------- packed weights
# mla_kv_prolog_prepare_weights: the decode kernel reads a re-laid-out copy
# of W_kva / W_kvb (bulk copies + TMA boxes of the hidden rows); same
# arithmetic, same tolerance against the oracle.

@pytest.mark.parametrize("b,s", [(1, 1), (1, 2), (4, 1), (8, 2), (32, 1), (64, 1), (64, 2), (128, 1)])
def test_packed_decode_v2lite(oracle_mod, b, s):
    r = run_case(I.V2_LITE, b, s, 700 + b * s, oracle_mod=oracle_mod, packed=True)
    assert r["status"] == 0


@pytest.mark.parametrize("T", [1, 17, 64, 100])
def test_packed_decode_r1(oracle_mod, T):
    r = run_case(I.R1, T, 1, 800 + T, oracle_mod=oracle_mod, packed=True)
    assert r["status"] == 0


@pytest.mark.parametrize("T", [3, 33, 127, 129, 200, 257])
def test_packed_ragged(oracle_mod, T):
    r = run_case(I.V2_LITE, T, 1, 900 + T, oracle_mod=oracle_mod, packed=True)
    tt = rows_per_launch(I.V2_LITE)
    assert r["status"] == 0 and r["launches"] == (T + tt - 1) // tt


@pytest.mark.parametrize("H,hidden,dtype", [(1, 64, "fp16"), (3, 192, "bf16"), (5, 640, "fp16"),
                                            (2, 2048, "bf16"), (16, 2048, "bf16"), (128, 2048, "fp16")])
def test_packed_small_shapes(oracle_mod, H, hidden, dtype):
    cfg = I.small_config(I.V2_LITE, hidden=hidden, num_heads=H, dtype=dtype)
    r = run_case(cfg, 3, 2, 950 + H, oracle_mod=oracle_mod, packed=True)
    assert r["status"] == 0


def test_packed_matches_raw_bitwise():
    """Same products in the same order: the packed and raw layouts give
    identical outputs."""
    a = run_case(I.V2_LITE, 16, 2, 4242)
    b = run_case(I.V2_LITE, 16, 2, 4242, packed=True)
    for k in ("k_nope", "value", "k_pe"):
        assert torch.equal(a["out"][k].view(torch.int16), b["out"][k].view(torch.int16)), k


def test_packed_snapshot_only_serves_its_own_weights(oracle_mod):
    """A run with other weight tensors reads them as passed; changing the
    snapshotted weights in place needs a new prepare; (None, None) forgets."""
    cfg = I.V2_LITE
    inp1 = I.kv_inputs(cfg, 4, 1, 11)
    inp2 = I.kv_inputs(cfg, 4, 1, 12)
    d1, d2 = B.to_device(inp1), B.to_device(inp2)
    m = B.MLAProlog(cfg, 4)
    m.set_path(B.PATH_DECODE)
    m.prepare_weights(d1)
    out = m.alloc_outputs(4, 1)
    m.run(4, 1, d2, out)  # other weights: raw path
    torch.cuda.synchronize()
    ref2 = oracle_mod.kv_prolog(inp2)
    for name, r in zip(("k_nope", "value", "k_pe"), ref2):
        compare(name, out[name], r, oracle_mod)
    m.run(4, 1, d1, out)  # snapshot
    torch.cuda.synchronize()
    ref1 = oracle_mod.kv_prolog(inp1)
    for name, r in zip(("k_nope", "value", "k_pe"), ref1):
        compare(name, out[name], r, oracle_mod)
    # in-place change of the snapshotted tensors, then a new snapshot
    d1["W_kva"].copy_(d2["W_kva"])
    d1["W_kvb"].copy_(d2["W_kvb"])
    m.prepare_weights(d1)
    m.run(4, 1, dict(d2, W_kva=d1["W_kva"], W_kvb=d1["W_kvb"]), out)
    torch.cuda.synchronize()
    for name, r in zip(("k_nope", "value", "k_pe"), ref2):
        compare(name, out[name], r, oracle_mod)
    B.mla_kv_prolog_prepare_weights(m.h, cfg, None, None)
    m.run(4, 1, d2, out)
    torch.cuda.synchronize()
    assert m.status() == 0
    m.close()


# ---------------------------------------------------------------- CUDA graphs
# A replayed graph re-runs the captured launch with the same arguments and
# workspace: the grid-barrier counters must be back at zero after each
# replay, and nothing a replay reads (split-K partials, latent rows) may be
# taken from the previous replay.  New hidden rows and positions are copied
# into the captured buffers before each replay; a replay that read the
# previous replay's partials would give the previous input's kv rows.

@pytest.mark.parametrize("cfg,b,packed", [(I.V2_LITE, 2, False), (I.V2_LITE, 16, True),
                                          (I.V2_LITE, 128, False), (I.R1, 64, True)])
def test_graph_replays_read_their_own_partials(oracle_mod, cfg, b, packed):
    inp = I.kv_inputs(cfg, b, 1, 900 + b)
    d = B.to_device(inp)
    m = B.MLAProlog(cfg, b)
    m.set_path(B.PATH_DECODE)
    if packed:
        m.prepare_weights(d)
    out = m.alloc_outputs(b, 1)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        m.run(b, 1, d, out, stream=st)  # first call outside capture
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            m.run(b, 1, d, out, stream=st)
    torch.cuda.synchronize()
    for rep in range(3):
        new = I.kv_inputs(cfg, b, 1, 950 + 10 * b + rep)
        d["hidden"].copy_(new["hidden"])
        d["positions"].copy_(new["positions"])
        for t in out.values():
            t.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert m.status() == 0
        ref = oracle_mod.kv_prolog(dict(inp, hidden=new["hidden"], positions=new["positions"]))
        for name, r in zip(("k_nope", "value", "k_pe"), ref):
            compare(name, out[name], r, oracle_mod)
    m.close()
