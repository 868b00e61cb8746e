"""GPU checks of the W8A8 full MLA prolog (through the C ABI).

Bit-exact: the per-row int8 quantisation of bf16 rows and the int8 GEMM
accumulators (against the oracle's brute-force integer GEMM), including the
split-K path; the q_b / kv_b accumulators computed from the GPU's own int8
operands.  Within tolerance: the five bf16 outputs against the fp64 oracle
(tiny shapes, R1 shapes at T = 1, 64 and sampled rows of T = 8192)."""
import numpy as np
import pytest
import torch

from mla_attention_kv_gb300 import binding as B
from mla_attention_kv_gb300 import build as BLD
from mla_attention_kv_gb300 import inputs as I

from parity import compare

pytestmark = pytest.mark.gpu
NAMES = ("q_nope", "q_pe", "k_nope", "value", "k_pe")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    BLD.build()
    B.load()


@pytest.mark.parametrize("rows,cols", [(1, 64), (7, 7168), (33, 1536), (3, 512), (5, 8184), (3, 8200)])
def test_quant_rows_bit_exact(oracle_mod, rows, cols):
    g = torch.Generator().manual_seed(rows * 1000 + cols)
    x = (torch.randn(rows, cols, generator=g) * 3).to(torch.bfloat16)
    x[0, :8] = torch.tensor([1.0, -2.0, 0.5, 0.0, 0.25, -0.125, 2.0, 1.5]).to(torch.bfloat16)
    if rows > 2:
        x[2] = 0  # amax == 0 row
    q = torch.empty(rows, cols, dtype=torch.int8, device="cuda")
    s = torch.empty(rows, dtype=torch.float32, device="cuda")
    B.mla_w8a8_quant_rows(x.cuda(), q, s)
    torch.cuda.synchronize()
    for r in range(rows):
        qo, so = oracle_mod.quant_row_f32(x[r].float().numpy())
        assert np.array_equal(q[r].cpu().numpy(), qo), r
        assert s[r].item() == so, r


@pytest.mark.parametrize("M,K,N", [(1, 7168, 1536), (1, 7168, 576), (64, 1536, 2048), (5, 512, 64),
                                   (130, 256, 192), (8192, 64, 64),
                                   # M <= 8: full-K TMA GEMV (K <= 2048) and split-K TMA GEMV
                                   (1, 1536, 24576), (8, 512, 32768), (3, 192, 384), (2, 64, 128),
                                   (7, 4096, 2112), (4, 2048, 320), (6, 2080, 64)])
def test_gemm_s32_bit_exact(oracle_mod, M, K, N):
    g = torch.Generator().manual_seed(M + K + N)
    A = torch.randint(-127, 128, (M, K), generator=g, dtype=torch.int8)
    W = torch.randint(-127, 128, (K, N), generator=g, dtype=torch.int8)
    acc = torch.empty(M, N, dtype=torch.int32, device="cuda")
    B.mla_w8a8_gemm_s32(A.cuda(), W.cuda(), acc)
    torch.cuda.synchronize()
    rows = np.unique(np.linspace(0, M - 1, min(M, 40)).astype(int))
    ref = oracle_mod.int_gemm(A.numpy()[rows], W.numpy())
    assert np.array_equal(acc.cpu().numpy()[rows].astype(np.int64), ref)


def run_w8(cfg, b, s, seed, positions="decode", rows=None, oracle_mod=None, keep=False):
    inp = I.w8a8_inputs(cfg, b, s, seed, positions)
    d = B.to_device(inp)
    m = B.MLAProlog(cfg, b * s)
    out = m.alloc_outputs(b, s)
    for t in out.values():
        t.fill_(float("nan"))
    m.run(b, s, d, out)
    torch.cuda.synchronize()
    st = m.status()
    res = dict(inp=inp, d=d, out=out, status=st, launches=m.last_launches, m=m)
    if oracle_mod is not None:
        ref = oracle_mod.w8a8_prolog(inp, rows=rows)
        res["err"] = {n: compare(n, out[n], r, oracle_mod) for n, r in zip(NAMES, ref)}
    if not keep:
        m.close()
    return res


def test_w8a8_tiny(oracle_mod):
    cfg = I.small_config(I.R1_W8A8, hidden=256, q_lora_rank=192, num_heads=2, max_pos=64)
    r = run_w8(cfg, 1, 3, 21, oracle_mod=oracle_mod)
    assert r["status"] == 0


@pytest.mark.parametrize("b,s", [(1, 1), (64, 1), (2, 1), (1, 2), (5, 1), (4, 2)])
def test_w8a8_r1_decode(oracle_mod, b, s):
    r = run_w8(I.R1_W8A8, b, s, I.seed_for(4) + b, oracle_mod=oracle_mod)
    assert r["status"] == 0


def test_w8a8_r1_prefill_sampled(oracle_mod):
    b, s = 1, 8192
    rows = I.tile_rows(b, s, 512, seed=2004)
    r = run_w8(I.R1_W8A8, b, s, I.seed_for(4), positions="prefill", rows=rows, oracle_mod=oracle_mod)
    assert r["status"] == 0


@pytest.mark.parametrize("b", [16, 4])
def test_w8a8_operands_and_accumulators(oracle_mod, b):
    """The int8 operands the GPU fed to q_b / kv_b agree with the oracle's
    requantisation (>= 99.9 % equal, never off by more than 1), and the
    int32 accumulators the GPU GEMM forms from them are bit-exact.  b = 4
    runs the decode-size chain (fused quantisation, split-K GEMV)."""
    cfg = I.R1_W8A8
    s = 1
    r = run_w8(cfg, b, s, 4242, keep=True)
    m, T = r["m"], b * s
    rq = cfg["q_lora_rank"]
    q1 = torch.empty(T, rq, dtype=torch.int8, device="cuda")
    s1 = torch.empty(T, dtype=torch.float32, device="cuda")
    c1 = torch.empty(T, 512, dtype=torch.int8, device="cuda")
    s2 = torch.empty(T, dtype=torch.float32, device="cuda")
    B.mla_prolog_w8a8_operands(m.h, T, q1, s1, c1, s2)
    torch.cuda.synchronize()
    m.close()
    gq, gc = q1.cpu().numpy(), c1.cpu().numpy()
    eq = tot = 0
    for t in range(T):
        oq, os1, oc, os2 = oracle_mod.w8a8_operands(r["inp"], t)
        for g_, o_ in ((gq[t], oq), (gc[t], oc)):
            d = np.abs(g_.astype(np.int32) - o_.astype(np.int32))
            assert d.max() <= 1
            eq += int((d == 0).sum())
            tot += d.size
        assert abs(s1[t].item() - os1) <= 1e-6 * os1 and abs(s2[t].item() - os2) <= 1e-6 * os2
    assert eq / tot >= 0.999, eq / tot
    # accumulators of the GPU's own operands: bit-exact against brute force
    for A, W in ((q1, r["d"]["W_qb"]), (c1, r["d"]["W_kvb"])):
        acc = torch.empty(T, W.shape[1], dtype=torch.int32, device="cuda")
        B.mla_w8a8_gemm_s32(A, W, acc)
        torch.cuda.synchronize()
        ref = oracle_mod.int_gemm(A.cpu().numpy()[:4], W.cpu().numpy())
        assert np.array_equal(acc.cpu().numpy()[:4].astype(np.int64), ref)


def test_w8a8_small_chain_repeats_and_alternates(oracle_mod):
    """The decode-size chain adds split-K partials into accumulator rows that
    the previous call left zeroed: repeated calls, and a prefill-size call in
    between, give the same outputs."""
    cfg = I.small_config(I.R1_W8A8, hidden=512, q_lora_rank=256, num_heads=4, max_pos=64)
    inp = I.w8a8_inputs(cfg, 3, 1, 77, "decode")
    d = B.to_device(inp)
    big = I.w8a8_inputs(cfg, 2, 16, 78, "prefill")
    db = B.to_device(big)
    m = B.MLAProlog(cfg, 64)
    try:
        outs = []
        for i in range(3):
            out = m.alloc_outputs(3, 1)
            m.run(3, 1, d, out)
            torch.cuda.synchronize()
            outs.append({k: v.clone() for k, v in out.items()})
            ob = m.alloc_outputs(2, 16)
            m.run(2, 16, db, ob)
            torch.cuda.synchronize()
        assert m.status() == 0
        for o in outs[1:]:
            for k in NAMES:
                assert torch.equal(o[k], outs[0][k]), k
        ref = oracle_mod.w8a8_prolog(inp)
        for n, r in zip(NAMES, ref):
            compare(n, outs[0][n], r, oracle_mod)
    finally:
        m.close()


def test_w8a8_paths_alternate_on_one_handle(oracle_mod):
    """All three W8A8 paths on one handle, twice in a row: the 2-SM path
    (T = 600, which stores its q_a | kv_a sums and leaves only the rows that
    smaller calls use zeroed), the single-SM path (T = 64) and the
    decode-size chain (T = 3), which both add into accumulator rows the call
    before left zeroed.  Every call matches the oracle and its repetition."""
    cfg = I.small_config(I.R1_W8A8, hidden=512, q_lora_rank=256, num_heads=4, max_pos=512)
    sizes = [(2, 300), (64, 1), (3, 1)]
    inps = [I.w8a8_inputs(cfg, b, s, 7100 + b * s, "decode") for b, s in sizes]
    devs = [B.to_device(x) for x in inps]
    m = B.MLAProlog(cfg, 600)
    try:
        rounds = []
        for _ in range(2):
            outs = []
            for (b, s), d in zip(sizes, devs):
                out = m.alloc_outputs(b, s)
                m.run(b, s, d, out)
                torch.cuda.synchronize()
                outs.append({k: v.clone() for k, v in out.items()})
            rounds.append(outs)
        assert m.status() == 0
        for o0, o1 in zip(*rounds):
            for k in NAMES:
                assert torch.equal(o0[k], o1[k]), k
        for inp, o in zip(inps, rounds[0]):
            for n, r in zip(NAMES, oracle_mod.w8a8_prolog(inp)):
                compare(n, o[n], r, oracle_mod)
    finally:
        m.close()


def _capture_run(cfg, inp, b, s):
    """Run the W8A8 prolog on `inp` with the accumulator capture on; return
    the captured accumulators and the GPU's own q_b / kv_b operands."""
    T, H, rq = b * s, cfg["num_heads"], cfg["q_lora_rank"]
    d = B.to_device(inp)
    m = B.MLAProlog(cfg, T)
    try:
        cap_a = torch.full((T, rq + 576), -7, dtype=torch.int32, device="cuda")
        cap_qb = torch.full((T, H * 192), -7, dtype=torch.int32, device="cuda")
        cap_kvb = torch.full((T, H * 256), -7, dtype=torch.int32, device="cuda")
        B.mla_prolog_w8a8_capture(m.h, cap_a, cap_qb, cap_kvb)
        out = m.alloc_outputs(b, s)
        m.run(b, s, d, out)
        q1 = torch.empty(T, rq, dtype=torch.int8, device="cuda")
        s1 = torch.empty(T, dtype=torch.float32, device="cuda")
        c1 = torch.empty(T, 512, dtype=torch.int8, device="cuda")
        s2 = torch.empty(T, dtype=torch.float32, device="cuda")
        B.mla_prolog_w8a8_operands(m.h, T, q1, s1, c1, s2)
        torch.cuda.synchronize()
        assert m.status() == 0
        B.mla_prolog_w8a8_capture(m.h)
    finally:
        m.close()
    return cap_a, cap_qb, cap_kvb, q1, c1


def _check_captured(oracle_mod, inp, caps, rows):
    cap_a, cap_qb, cap_kvb, q1, c1 = caps
    hid = inp["hidden"].float().numpy()
    qx = np.stack([oracle_mod.quant_row_f32(hid[t])[0] for t in rows])
    w_a = np.concatenate([inp["W_qa"].numpy(), inp["W_kva"].numpy()], axis=1)
    assert np.array_equal(cap_a.cpu().numpy()[rows].astype(np.int64), oracle_mod.int_gemm(qx, w_a))
    for cap, A, W in ((cap_qb, q1, inp["W_qb"]), (cap_kvb, c1, inp["W_kvb"])):
        ref = oracle_mod.int_gemm(A.cpu().numpy()[rows], W.numpy())
        assert np.array_equal(cap.cpu().numpy()[rows].astype(np.int64), ref)


@pytest.mark.parametrize("pattern", ["all_max", "random_signs", "full_range"])
@pytest.mark.parametrize("b,s", [(64, 1), (3, 5), (2, 300)])
def test_w8a8_accumulators_adversarial(oracle_mod, pattern, b, s):
    """Inputs that push the exact-integer argument of the tensor-core paths
    to its limit: every code +127 (each fp32 chunk sum reaches 512 * 127^2
    on the single-SM kernel, T = 64 and 15, and 1024 * 127^2 < 2^24 on the
    2-SM kernel, T = 600), the same magnitudes with random signs, and
    full-range random int8 weights; the captured int32 accumulators of all
    four GEMMs stay bit-exact."""
    cfg = I.R1_W8A8
    T = b * s
    inp = I.w8a8_inputs(cfg, b, s, 6000 + T, "decode")
    g = torch.Generator().manual_seed(6100 + T)
    wk = ("W_qa", "W_kva", "W_qb", "W_kvb")
    if pattern == "all_max":
        inp["hidden"] = torch.ones_like(inp["hidden"])  # every code +127
        for k in wk:
            inp[k] = torch.full_like(inp[k], 127)
    elif pattern == "random_signs":
        inp["hidden"] = (torch.randint(0, 2, inp["hidden"].shape, generator=g) * 2 - 1).to(torch.bfloat16)
        for k in wk:
            inp[k] = ((torch.randint(0, 2, inp[k].shape, generator=g) * 2 - 1) * 127).to(torch.int8)
    else:
        inp["hidden"] = (torch.randn(inp["hidden"].shape, generator=g) * 3).to(torch.bfloat16)
        for k in wk:
            inp[k] = torch.randint(-127, 128, inp[k].shape, generator=g, dtype=torch.int8)
    caps = _capture_run(cfg, inp, b, s)
    _check_captured(oracle_mod, inp, caps, sorted({0, T // 2, T - 1}))


@pytest.mark.parametrize("b,s", [(1, 1), (2, 1), (4, 1), (8, 1), (64, 1), (3, 33), (1, 8192)])
def test_w8a8_run_accumulators_bit_exact(oracle_mod, b, s):
    """The int32 accumulators that the run's own kernels formed (captured
    from the kernels of the call: the decode-size chain at T <= 8, the
    prefill-size path above), bit for bit against the oracle's brute-force
    integer GEMM ([R1] §权重转换, W8A8: int32 accumulation is exact).
    q_a | kv_a: the oracle quantises the bf16 hidden rows itself (the codes
    are bit-identical on both sides).  q_b, kv_b: the operands are the
    GPU's own requantised rows (they may differ from the oracle's by one
    code at rounding ties, which the operand test bounds)."""
    cfg = I.R1_W8A8
    T = b * s
    inp = I.w8a8_inputs(cfg, b, s, 5150 + T, "decode" if s == 1 else "prefill")
    caps = _capture_run(cfg, inp, b, s)
    _check_captured(oracle_mod, inp, caps, sorted({0, T - 1, T // 2, min(1, T - 1)}))
