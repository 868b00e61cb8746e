"""GPU parity of the cluster decode kernel (launches of at most 16 rows on the
packed snapshot, V2-Lite shape) against the fp64 oracle, through the C ABI:
every row count from 1 to 16 in both dtypes, head counts that leave CTAs
without kv_b columns, paged outputs, back-to-back calls of mixed sizes
chained with the grid-barrier kernel, a replayed CUDA graph, the bounded
device waits, and the cases that must not take it."""
import pytest
import torch

from mla_attention_kv_gb300 import binding as B
from mla_attention_kv_gb300 import build as BLD
from mla_attention_kv_gb300 import inputs as I

from parity import compare

pytestmark = pytest.mark.gpu
KV = ("k_nope", "value", "k_pe")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    BLD.build()
    B.load()


def run_packed(cfg, b, s, seed, path=B.PATH_DECODE, oracle_mod=None, spin_budget_ns=0, positions="decode"):
    inp = I.kv_inputs(cfg, b, s, seed, positions)
    d = B.to_device(inp)
    m = B.MLAProlog(cfg, b * s, spin_budget_ns=spin_budget_ns)
    m.set_path(path)
    m.prepare_weights(d)
    out = m.alloc_outputs(b, s)
    for t in out.values():
        t.fill_(float("nan"))
    m.run(b, s, d, out)
    torch.cuda.synchronize()
    res = dict(inp=inp, out=out, status=m.status(), launches=m.last_launches,
               cl=m.last_cluster_launches, path=m.last_path)
    if oracle_mod is not None:
        ref = oracle_mod.kv_prolog(inp)
        for name, r in zip(KV, ref):
            compare(name, out[name], r, oracle_mod)
    m.close()
    return res


@pytest.mark.parametrize("T", list(range(1, 17)))
def test_cluster_rows_fp16(oracle_mod, T):
    r = run_packed(I.V2_LITE, T, 1, 1200 + T, oracle_mod=oracle_mod)
    assert r["status"] == 0 and r["launches"] == 1 and r["cl"] == 1 and r["path"] == B.PATH_DECODE


@pytest.mark.parametrize("b,s", [(1, 1), (1, 2), (3, 2), (8, 2), (16, 1)])
def test_cluster_rows_bf16(oracle_mod, b, s):
    cfg = I.small_config(I.V2_LITE, dtype="bf16")
    r = run_packed(cfg, b, s, 1300 + b * s, oracle_mod=oracle_mod)
    assert r["status"] == 0 and r["cl"] == 1


@pytest.mark.parametrize("H", [1, 2, 7, 17])
def test_cluster_head_counts(oracle_mod, H):
    # few heads: most CTAs own no kv_b columns; 17 heads: the widest slices that fit
    cfg = I.small_config(I.V2_LITE, num_heads=H)
    r = run_packed(cfg, 5, 1, 1400 + H, oracle_mod=oracle_mod)
    assert r["status"] == 0 and r["cl"] == 1


def test_cluster_prefill_positions(oracle_mod):
    # s = 16 consecutive positions of one sequence (the rows of one launch)
    r = run_packed(I.V2_LITE, 1, 16, 1450, oracle_mod=oracle_mod, positions="prefill")
    assert r["status"] == 0 and r["cl"] == 1


def test_cluster_not_taken():
    cfg = I.V2_LITE
    # more rows than the kernel takes, the forced grid kernel, raw weights
    assert run_packed(cfg, 17, 1, 1500)["cl"] == 0
    assert run_packed(cfg, 4, 1, 1501, path=B.PATH_DECODE_GRID)["cl"] == 0
    inp = I.kv_inputs(cfg, 4, 1, 1502)
    d = B.to_device(inp)
    m = B.MLAProlog(cfg, 4)
    out = m.alloc_outputs(4, 1)
    m.run(4, 1, d, out)
    torch.cuda.synchronize()
    assert m.status() == 0 and m.last_cluster_launches == 0
    m.close()
    # another hidden size (R1); column slices wider than the shared memory holds
    assert run_packed(I.R1, 8, 1, 1503)["cl"] == 0
    assert run_packed(I.small_config(I.V2_LITE, num_heads=32), 8, 1, 1504)["cl"] == 0


def test_cluster_matches_grid_kernel(oracle_mod):
    """Both decode kernels stay within the oracle tolerance on the same inputs,
    and agree with each other to within two steps of the dtype grid plus
    2e-3 absolute (the fp32 sums are taken in other orders, so a latent value
    may round the other way and move outputs near zero by about 1e-4)."""
    a = run_packed(I.V2_LITE, 8, 2, 1600, oracle_mod=oracle_mod)
    g = run_packed(I.V2_LITE, 8, 2, 1600, path=B.PATH_DECODE_GRID, oracle_mod=oracle_mod)
    assert a["cl"] == 1 and g["cl"] == 0
    for k in KV:
        x, y = a["out"][k].float(), g["out"][k].float()
        step = torch.maximum(x.abs(), y.abs()) * 2.0 ** -9 + 2e-3
        assert torch.all((x - y).abs() <= step), k


def test_cluster_deterministic():
    a = run_packed(I.V2_LITE, 16, 1, 1700)
    b = run_packed(I.V2_LITE, 16, 1, 1700)
    for k in KV:
        assert torch.equal(a["out"][k].view(torch.int16), b["out"][k].view(torch.int16)), k


def test_chained_calls_mixed_sizes(oracle_mod):
    """Calls of 1 .. 128 rows back to back on one stream, each chained to the
    previous launch (cluster and grid-barrier kernels alternate), every
    output checked afterwards."""
    cfg = I.V2_LITE
    sizes = [1, 16, 32, 4, 128, 8, 2, 64, 16, 3]
    inp0 = I.kv_inputs(cfg, max(sizes), 1, 1800)
    d0 = B.to_device(inp0)
    m = B.MLAProlog(cfg, max(sizes))
    m.prepare_weights(d0)
    torch.cuda.synchronize()
    runs = []
    for i, T in enumerate(sizes):
        inp = I.kv_inputs(cfg, T, 1, 1810 + i)
        d = B.to_device(inp)
        d.update(W_kva=d0["W_kva"], W_kvb=d0["W_kvb"], gamma_kv=d0["gamma_kv"])
        inp.update(W_kva=inp0["W_kva"], W_kvb=inp0["W_kvb"], gamma_kv=inp0["gamma_kv"])
        out = m.alloc_outputs(T, 1)
        for t in out.values():
            t.fill_(float("nan"))
        runs.append((T, inp, d, out))
    torch.cuda.synchronize()
    cls = []
    for T, inp, d, out in runs:
        m.run(T, 1, d, out)
        cls.append(m.last_cluster_launches)
    torch.cuda.synchronize()
    assert m.status() == 0
    assert cls == [1 if T <= 16 else 0 for T in sizes]
    for T, inp, d, out in runs:
        ref = oracle_mod.kv_prolog(inp)
        for name, r in zip(KV, ref):
            compare(name, out[name], r, oracle_mod)
    m.close()


def test_cluster_graph_replay(oracle_mod):
    cfg, b = I.V2_LITE, 12
    inp = I.kv_inputs(cfg, b, 1, 1900)
    d = B.to_device(inp)
    m = B.MLAProlog(cfg, b)
    m.prepare_weights(d)
    out = m.alloc_outputs(b, 1)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        m.run(b, 1, d, out, stream=st)
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            for _ in range(3):  # three chained launches per replay
                m.run(b, 1, d, out, stream=st)
    torch.cuda.synchronize()
    assert m.last_cluster_launches == 1
    for rep in range(3):
        new = I.kv_inputs(cfg, b, 1, 1910 + rep)
        d["hidden"].copy_(new["hidden"])
        d["positions"].copy_(new["positions"])
        for t in out.values():
            t.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert m.status() == 0
        ref = oracle_mod.kv_prolog(dict(inp, hidden=new["hidden"], positions=new["positions"]))
        for name, r in zip(KV, ref):
            compare(name, out[name], r, oracle_mod)
    m.close()


def test_cluster_paged(oracle_mod):
    from test_paged_gpu import make_slots, run_paged
    b, s, page, nblk = 6, 2, 4, 8
    slots = make_slots(b * s, page, nblk, 21, drop=(2, 9))
    assert run_paged(I.V2_LITE, b, s, 2000, page, nblk, slots, B.PATH_DECODE, oracle_mod=oracle_mod,
                     packed=True) == 0


def test_cluster_bad_position_is_flagged(oracle_mod):
    cfg = I.V2_LITE
    inp = I.kv_inputs(cfg, 4, 1, 2100, positions=[5, 4096, -3, 100])
    d = B.to_device(inp)
    m = B.MLAProlog(cfg, 4)
    m.prepare_weights(d)
    out = m.alloc_outputs(4, 1)
    m.run(4, 1, d, out)
    torch.cuda.synchronize()
    assert m.last_cluster_launches == 1 and m.status() == 7
    m.close()
    ref = oracle_mod.kv_prolog(dict(inp, positions=torch.tensor([5, 0, 0, 100], dtype=torch.int32)))
    compare("k_nope", out["k_nope"], ref[0], oracle_mod)
    compare("k_pe", out["k_pe"][[0, 3]], ref[2][[0, 3]], oracle_mod)


def test_cluster_wait_budget_expires_cleanly():
    """A 1 ns wait budget: the CTAs give up on their copies, still send both
    rounds, wait for what is in flight and leave; the call reports
    MLA_ERR_DEVICE_TIMEOUT and a normal handle is correct afterwards."""
    r = run_packed(I.V2_LITE, 4, 1, 2200, spin_budget_ns=1)
    assert r["cl"] == 1 and r["status"] == 6
    r = run_packed(I.V2_LITE, 4, 1, 2200)
    assert r["status"] == 0 and r["cl"] == 1
