"""Pins of the CPU oracle to facts outside itself (CPU only).

Each test ties one part of the oracle to something it does not compute
itself: exhaustive checks of the 16-bit encodings against numpy / torch
decoders and against the round-to-nearest-even definition, closed forms
and hand-derived values (tests/golden), invariants of RMSNorm and RoPE,
integer-exact matmuls, and routing weights whose outputs are known in
closed form.  A dropped term, a wrong sign, a wrong index or a transposed
operand in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from mla_attention_kv_gb300 import inputs as I

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ------------------------------------------------------------ 16-bit encodings
def test_f16_decode_exhaustive(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle_mod.promote16(bits, 0)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])
    assert np.array_equal(np.signbit(ref[m]), np.signbit(got[m]))


def test_bf16_decode_exhaustive(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = oracle_mod.promote16(bits, 1)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])


@pytest.mark.parametrize("dtype", [0, 1])
def test_encode_roundtrip_and_ties(oracle_mod, dtype):
    """Every finite value encodes to itself; each midpoint between adjacent
    values goes to the one with an even last fraction bit, and a nudge off
    the midpoint goes to the nearer one (definition of RNE)."""
    enc = oracle_mod.double_to_f16 if dtype == 0 else oracle_mod.double_to_bf16
    ebits = 5 if dtype == 0 else 8
    mant = 10 if dtype == 0 else 7
    top = ((1 << ebits) - 1) << mant  # +inf pattern
    pos = np.arange(0, top + 1, dtype=np.uint32).astype(np.uint16)  # +0 .. +inf
    vals = oracle_mod.promote16(pos, dtype)
    for bb, v in zip(pos[::7].tolist(), vals[::7].tolist()):
        assert enc(v) == bb
        assert enc(-v) == (bb | 0x8000)
    # midpoints between every adjacent pair of finite positive values
    lo, hi = vals[:-2], vals[1:-1]
    lob, hib = pos[:-2], pos[1:-1]
    for i in range(0, lo.size, 13):
        mid = (lo[i] + hi[i]) / 2.0  # exact in double
        even = lob[i] if (int(lob[i]) & 1) == 0 else hib[i]
        assert enc(mid) == even
        assert enc(mid + (hi[i] - lo[i]) * 1e-6) == hib[i]
        assert enc(mid - (hi[i] - lo[i]) * 1e-6) == lob[i]
    # overflow threshold: halfway above the largest finite value ties to inf
    maxfin = vals[-2]
    step = vals[-2] - vals[-3]
    assert enc(maxfin + step / 2) == top
    assert enc(maxfin + step / 2 * (1 - 1e-9)) == pos[-2]


def test_f16_encode_matches_numpy(oracle_mod):
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000),
                        rng.standard_normal(500) * 1e-6])
    ref = x.astype(np.float16).view(np.uint16)
    got = np.array([oracle_mod.double_to_f16(v) for v in x], dtype=np.uint16)
    assert np.array_equal(ref, got)


def test_bf16_encode_matches_torch_on_float32_inputs(oracle_mod):
    rng = np.random.default_rng(8)
    x = (rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle_mod.double_to_bf16(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(ref, got)


# ------------------------------------------------------------ RMSNorm
def test_rmsnorm_hand_values(oracle_mod):
    g = _gold("rmsnorm_hand.json")
    for c in g["cases"]:
        pat = np.array(c["pattern"], dtype=np.float64)
        x = np.tile(pat, c["n"] // pat.size)
        y = oracle_mod.rmsnorm(x, np.full(c["n"], c["gamma"]), c["eps"])
        np.testing.assert_allclose(y[:2], c["expect_first_two"], rtol=1e-15, atol=0)


def test_rmsnorm_constant_closed_form(oracle_mod):
    for cval in (1e-4, 0.3, 7.0):
        gam = np.linspace(0.5, 1.5, 512)
        y = oracle_mod.rmsnorm(np.full(512, cval), gam, 1e-6)
        np.testing.assert_allclose(y, gam * cval / math.sqrt(cval * cval + 1e-6), rtol=1e-14)


def test_rmsnorm_invariants(oracle_mod):
    rng = np.random.default_rng(1)
    x = rng.standard_normal(512) * 3.0
    gam = 1.0 + 0.1 * rng.standard_normal(512)
    eps = 1e-6
    y = oracle_mod.rmsnorm(x, gam, eps)
    ms = float(np.mean(x * x))
    # mean((y / gamma)^2) = ms / (ms + eps)
    np.testing.assert_allclose(np.mean((y / gam) ** 2), ms / (ms + eps), rtol=1e-13)
    # sign of every entry follows x * gamma; scaling x (eps negligible) keeps y
    assert np.all(np.sign(y) == np.sign(x * gam))
    y2 = oracle_mod.rmsnorm(1024.0 * x, gam, eps)
    np.testing.assert_allclose(y2, y, rtol=1e-6)


# ------------------------------------------------------------ RoPE
def test_rope_hand_value(oracle_mod):
    g = _gold("rope_hand.json")
    cos, sin = I.rope_tables(8, 64, 10000.0)
    assert float(cos[1, 0]) == g["cos_f32"] and float(sin[1, 0]) == g["sin_f32"]
    x = np.zeros(64)
    x[0], x[1] = g["x0"], g["x1"]
    y = oracle_mod.rope(x, cos[g["position"]].numpy(), sin[g["position"]].numpy())
    assert y[0] == pytest.approx(g["expect_out0"], abs=1e-15)
    assert y[32] == pytest.approx(g["expect_out32"], abs=1e-15)
    assert np.count_nonzero(y) == 2


def test_rope_position_zero_is_deinterleave(oracle_mod):
    cos, sin = I.rope_tables(4, 64, 10000.0)
    x = np.arange(64, dtype=np.float64) + 0.25
    y = oracle_mod.rope(x, cos[0].numpy(), sin[0].numpy())
    assert np.array_equal(y, np.concatenate([x[0::2], x[1::2]]))


def test_rope_pair_norm_and_angle(oracle_mod):
    """Each pair (x[2j], x[2j+1]) is rotated, as (out[j], out[j+32]), by
    p * theta^(-2j/64): norm kept, angle advanced by exactly that much."""
    cos, sin = I.rope_tables(4096, 64, 10000.0)
    rng = np.random.default_rng(3)
    for p in (1, 17, 4095):
        x = rng.standard_normal(64)
        y = oracle_mod.rope(x, cos[p].numpy(), sin[p].numpy())
        for j in range(32):
            a, bb = x[2 * j], x[2 * j + 1]
            u, v = y[j], y[j + 32]
            assert u * u + v * v == pytest.approx(a * a + bb * bb, rel=2e-7)
            want = p * 10000.0 ** (-2.0 * j / 64)
            got = math.atan2(v, u) - math.atan2(bb, a)
            d = (got - want + math.pi) % (2 * math.pi) - math.pi
            assert abs(d) < 2e-6 * max(1.0, want)


def test_rope_relative_position(oracle_mod):
    cos, sin = I.rope_tables(64, 64, 10000.0)
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal(64), rng.standard_normal(64)

    def dot(m, n):
        return float(np.dot(oracle_mod.rope(q, cos[m].numpy(), sin[m].numpy()),
                            oracle_mod.rope(k, cos[n].numpy(), sin[n].numpy())))
    assert dot(5, 3) == pytest.approx(dot(12, 10), rel=1e-6, abs=1e-6)
    assert dot(40, 9) == pytest.approx(dot(31, 0), rel=1e-6, abs=1e-6)


def test_rope_tables_match_math(oracle_mod):
    cos, sin = I.rope_tables(4096, 64, 10000.0)
    for p in (0, 1, 100, 4095):
        for i in (0, 5, 31, 32, 63):
            ang = p * 10000.0 ** (-2.0 * (i % 32) / 64)
            assert float(cos[p, i]) == float(np.float32(math.cos(ang)))
            assert float(sin[p, i]) == float(np.float32(math.sin(ang)))


# ------------------------------------------------------------ matmul
def test_vec_matmul_integer_exact(oracle_mod):
    rng = np.random.default_rng(5)
    x = rng.integers(-8, 9, 37).astype(np.float64)
    W = rng.integers(-8, 9, (37, 23)).astype(np.float64)
    y = oracle_mod.vec_matmul(x, W)
    ref = (x.astype(np.int64) @ W.astype(np.int64)).astype(np.float64)
    assert np.array_equal(y, ref)


def test_vec_matmul_bruteforce(oracle_mod):
    rng = np.random.default_rng(6)
    x = rng.standard_normal(11)
    W = rng.standard_normal((11, 5))
    y = oracle_mod.vec_matmul(x, W)
    for n in range(5):  # k-outer brute force, written independently
        acc = math.fsum(x[k] * W[k, n] for k in range(11))
        assert y[n] == pytest.approx(acc, rel=1e-14, abs=1e-14)


# ------------------------------------------------------------ whole KV prolog
def _routing_case(b, s, H, positions, dtype="fp16"):
    """Closed-form case: W_kva = [I_576; 0] routes hidden[:, :576] to the
    kv_a output; each token's latent is c_t * sign pattern (RMSNorm known in
    closed form); W_kvb has one entry w_j per column at row src(j)."""
    cfg = I.small_config(I.V2_LITE, hidden=640, num_heads=H, dtype=dtype, max_pos=4096)
    dt = I.torch_dtype(cfg)
    T = b * s
    r, dr = 512, 64
    nb = H * 256
    sign = np.where(np.arange(r) % 3 == 0, -1.0, 1.0)
    cvals = np.array([0.5, 1.0, 2.0, 0.25, 4.0, 1.5, 3.0, 0.75] * 8)[:T]
    hid = np.zeros((T, 640))
    rng = np.random.default_rng(9)
    for t in range(T):
        hid[t, :r] = cvals[t] * sign
        hid[t, r:r + dr] = rng.integers(-16, 17, dr) / 8.0
        hid[t, r + dr:] = rng.standard_normal(640 - r - dr)  # must be ignored
    Wa = np.zeros((640, r + dr))
    Wa[np.arange(r + dr), np.arange(r + dr)] = 1.0
    gam = np.where(np.arange(r) % 2 == 0, 0.5, 2.0)
    src = (7 * np.arange(nb) + 3) % r
    wj = np.where(np.arange(nb) % 5 == 0, -0.25, 0.5)
    Wb = np.zeros((r, nb))
    Wb[src, np.arange(nb)] = wj
    cos, sin = I.rope_tables(4096, 64, 10000.0)
    inp = dict(cfg=cfg, b=b, s=s, hidden=torch.tensor(hid).to(dt), W_kva=torch.tensor(Wa).to(dt),
               gamma_kv=torch.tensor(gam).to(dt), W_kvb=torch.tensor(Wb).to(dt),
               positions=torch.tensor(positions, dtype=torch.int32), cos=cos, sin=sin)
    return inp, hid, sign, cvals, gam, src, wj


@pytest.mark.parametrize("b,s", [(2, 3), (1, 6), (6, 1)])
def test_kv_prolog_routing_closed_form(oracle_mod, b, s):
    H = 2
    T = b * s
    positions = [0, 5, 0, 99, 4095, 1][:T]
    inp, hid, sign, cvals, gam, src, wj = _routing_case(b, s, H, positions)
    k_nope, value, k_pe = oracle_mod.kv_prolog(inp, nthreads=1)
    assert k_nope.shape == (b, H, s, 128) and value.shape == (b, H, s, 128)
    assert k_pe.shape == (b, 1, s, 64)
    for t in range(T):
        bi, si = divmod(t, s)
        c = cvals[t]
        n = c * sign / math.sqrt(c * c + 1e-6) * gam  # RMSNorm closed form
        kv = wj * n[src]
        for hh in range(H):
            np.testing.assert_allclose(k_nope[bi, hh, si], kv[hh * 256:hh * 256 + 128], rtol=1e-14)
            np.testing.assert_allclose(value[bi, hh, si], kv[hh * 256 + 128:hh * 256 + 256],
                                       rtol=1e-14)
        raw = hid[t, 512:576]
        if positions[t] == 0:
            assert np.array_equal(k_pe[bi, 0, si], np.concatenate([raw[0::2], raw[1::2]]))
        else:
            for j in range(32):
                u, v = k_pe[bi, 0, si, j], k_pe[bi, 0, si, j + 32]
                assert u * u + v * v == pytest.approx(raw[2 * j] ** 2 + raw[2 * j + 1] ** 2,
                                                      rel=1e-6, abs=1e-12)
            # the (hand-pinned) RoPE of the raw columns at this token's position
            p = positions[t]
            want = oracle_mod.rope(raw, inp["cos"][p].numpy(), inp["sin"][p].numpy())
            np.testing.assert_allclose(k_pe[bi, 0, si], want, rtol=1e-14, atol=1e-15)


def test_kv_prolog_token_independence_and_sampling(oracle_mod):
    cfg = I.small_config(I.V2_LITE, hidden=128, num_heads=3)
    inp = I.kv_inputs(cfg, 2, 5, seed=11, positions="decode")
    full = oracle_mod.kv_prolog(inp, nthreads=2)
    rows = [0, 4, 7]
    part = oracle_mod.kv_prolog(inp, rows=rows, nthreads=1)
    for t in range(10):
        bi, si = divmod(t, 5)
        for a, bb in zip(full, part):
            if t in rows:
                assert np.array_equal(a[bi, :, si], bb[bi, :, si])
            else:
                assert np.all(np.isnan(bb[bi, :, si]))
    # the same token rows laid out as (b=10, s=1) give the same values
    inp2 = dict(inp, b=10, s=1)
    flat = oracle_mod.kv_prolog(inp2, nthreads=1)
    for t in range(10):
        bi, si = divmod(t, 5)
        assert np.array_equal(full[0][bi, :, si], flat[0][t, :, 0])
        assert np.array_equal(full[2][bi, 0, si], flat[2][t, 0, 0])


def test_kv_prolog_linearity(oracle_mod):
    """Doubling W_kvb doubles k_nope / value exactly and leaves k_pe; scaling
    the hidden row by 2 doubles k_pe and leaves k_nope up to eps."""
    cfg = I.small_config(I.V2_LITE, hidden=128, num_heads=2)
    inp = I.kv_inputs(cfg, 1, 3, seed=12, positions="decode")
    a = oracle_mod.kv_prolog(inp, nthreads=1)
    inp2 = dict(inp, W_kvb=(inp["W_kvb"].float() * 2).to(inp["W_kvb"].dtype))
    b2 = oracle_mod.kv_prolog(inp2, nthreads=1)
    assert np.array_equal(b2[0], 2 * a[0]) and np.array_equal(b2[1], 2 * a[1])
    assert np.array_equal(b2[2], a[2])
    inp3 = dict(inp, hidden=(inp["hidden"].float() * 2).to(inp["hidden"].dtype))
    c = oracle_mod.kv_prolog(inp3, nthreads=1)
    np.testing.assert_allclose(c[2], 2 * a[2], rtol=1e-12)
    np.testing.assert_allclose(c[0], a[0], rtol=1e-5, atol=1e-9)


def test_kv_prolog_bad_position(oracle_mod):
    cfg = I.small_config(I.V2_LITE, hidden=64, num_heads=1, max_pos=16)
    inp = I.kv_inputs(cfg, 1, 2, seed=1, positions=[3, 16])
    with pytest.raises(ValueError):
        oracle_mod.kv_prolog(inp, nthreads=1)


# ------------------------------------------------------------ latent-cache variant
@pytest.mark.parametrize("b,s", [(2, 3), (6, 1)])
def test_kv_latent_routing_closed_form(oracle_mod, b, s):
    """Identity routing: the latent row is RMSNorm of c_t * sign in closed
    form, and k_pe is the same roped row as the full prolog's."""
    T = b * s
    positions = [0, 5, 0, 99, 4095, 1][:T]
    inp, hid, sign, cvals, gam, src, wj = _routing_case(b, s, 2, positions)
    latent, k_pe = oracle_mod.kv_latent(inp, nthreads=1)
    assert latent.shape == (T, 512) and k_pe.shape == (b, 1, s, 64)
    full_kpe = oracle_mod.kv_prolog(inp, nthreads=1)[2]
    assert np.array_equal(k_pe, full_kpe)
    for t in range(T):
        c = cvals[t]
        np.testing.assert_allclose(latent[t], c * sign / math.sqrt(c * c + 1e-6) * gam, rtol=1e-14)


def test_kv_latent_feeds_kv_b(oracle_mod):
    """latent x W_kvb (a library matmul in fp64), reshaped per head, is the
    full prolog's k_nope / value; rows not asked for stay NaN."""
    cfg = I.small_config(I.V2_LITE, hidden=192, num_heads=3)
    b, s = 2, 3
    inp = I.kv_inputs(cfg, b, s, seed=21, positions="decode")
    latent, k_pe = oracle_mod.kv_latent(inp, nthreads=2)
    k_nope, value, kpe_full = oracle_mod.kv_prolog(inp, nthreads=2)
    Wb = inp["W_kvb"].double().numpy()
    kv = latent @ Wb
    for t in range(b * s):
        bi, si = divmod(t, s)
        for hh in range(3):
            np.testing.assert_allclose(kv[t, hh * 256:hh * 256 + 128], k_nope[bi, hh, si], rtol=1e-9, atol=1e-12)
            np.testing.assert_allclose(kv[t, hh * 256 + 128:hh * 256 + 256], value[bi, hh, si], rtol=1e-9, atol=1e-12)
    assert np.array_equal(k_pe, kpe_full)
    part, kp2 = oracle_mod.kv_latent(inp, rows=[1, 4], nthreads=1)
    assert np.array_equal(part[[1, 4]], latent[[1, 4]])
    assert np.all(np.isnan(part[[0, 2, 3, 5]])) and np.all(np.isnan(kp2[0, 0, 0]))


# ------------------------------------------------------------ int8 KV-cache codes
def test_quant_c8_hand_values(oracle_mod):
    """x / scale rounded half to even and clamped to [-127, 127]; the input
    is first rounded to the I/O dtype (fp16 here: 0.1 -> 0.0999755859375)."""
    x = np.array([[0.5, -1.0, 0.015, 0.025, 3.0, -3.0, 0.1, 0.0]])
    sc = np.array([0.01, 0.01, 0.01, 0.01, 0.01, 0.01, 0.001, 0.5], dtype=np.float32)
    q = oracle_mod.quant_c8(x, sc, 0)
    # 0.015 and 0.025 in fp16 are 0.01499938965 and 0.02499389648: 1.4999 -> 1, 2.4994 -> 2
    assert q.tolist() == [[50, -100, 1, 2, 127, -127, 100, 0]]
    # exact ties go to even: 2.5 -> 2, 3.5 -> 4, -0.5 -> 0 (bf16 holds these exactly)
    q2 = oracle_mod.quant_c8(np.array([2.5, 3.5, -0.5, 1.5]), np.ones(4, dtype=np.float32), 1)
    assert q2.tolist() == [2, 4, 0, 2]


# ------------------------------------------------------------ paged KV-cache layout
def test_scatter_paged_identity_and_permutation(oracle_mod):
    """One block per sequence (slot = bi*s + si, page = s) reproduces the
    dense layout exactly; a permuted block table moves whole rows, and
    dropped rows (slot -1) leave NaN."""
    cfg = I.small_config(I.V2_LITE, hidden=128, num_heads=2)
    b, s = 3, 4
    inp = I.kv_inputs(cfg, b, s, seed=31, positions="decode")
    dense = oracle_mod.kv_prolog(inp, nthreads=1)
    same = oracle_mod.scatter_paged(dense, b, s, np.arange(b * s), s, b)
    for a, c in zip(dense, same):
        assert np.array_equal(a, c)
    page, nblk = 2, 9
    slots = np.array([17, 3, 4, 0, -1, 9, 10, 6, 1, 12, 13, -1])
    paged = oracle_mod.scatter_paged(dense, b, s, slots, page, nblk)
    written = set()
    for t in range(b * s):
        bi, si = divmod(t, s)
        if slots[t] < 0:
            continue
        blk, off = divmod(int(slots[t]), page)
        written.add((blk, off))
        for a, c in zip(dense, paged):
            assert np.array_equal(c[blk, :, off], a[bi, :, si])
    for blk in range(nblk):
        for off in range(page):
            if (blk, off) not in written:
                assert all(np.all(np.isnan(c[blk, :, off])) for c in paged)


# ------------------------------------------------------------ W8A8
def test_quant_hand_values(oracle_mod):
    for c in _gold("quant_hand.json")["cases"]:
        q, s = oracle_mod.quant_row_f32(np.array(c["x"], dtype=np.float32))
        assert q.tolist() == c["q"]
        assert s == c["scale"]


def test_quant_roundtrip_bound(oracle_mod):
    rng = np.random.default_rng(13)
    x = (rng.standard_normal(7168) * 2).astype(np.float32)
    q, s = oracle_mod.quant_row_f32(x)
    assert np.abs(q).max() == 127 and np.abs(q).min() >= 0
    # dequantisation error of symmetric rounding is at most half a step
    assert np.all(np.abs(q.astype(np.float64) * s - x) <= 0.5 * s * (1 + 1e-6))


def test_int_gemm_matches_integer_matmul(oracle_mod):
    rng = np.random.default_rng(14)
    A = rng.integers(-127, 128, (5, 300)).astype(np.int8)
    W = rng.integers(-127, 128, (300, 17)).astype(np.int8)
    acc = oracle_mod.int_gemm(A, W)
    assert np.array_equal(acc, A.astype(np.int64) @ W.astype(np.int64))
    # transposition check: a single non-zero weight lands in its own column
    W2 = np.zeros((300, 17), dtype=np.int8)
    W2[10, 3] = 1
    acc2 = oracle_mod.int_gemm(A, W2)
    assert np.array_equal(acc2[:, 3], A[:, 10].astype(np.int64))
    assert np.count_nonzero(acc2[:, np.arange(17) != 3]) == 0


def _tiny_w8_cfg():
    return I.small_config(I.R1_W8A8, hidden=256, q_lora_rank=192, num_heads=2, max_pos=64)


def test_w8a8_routing_q_side(oracle_mod):
    """One-hot W_qb: q_nope / q_pe pick the oracle's own requantised q
    operand at src(j), scaled by s1 * s_qb[j]; q_pe additionally rotated."""
    cfg = _tiny_w8_cfg()
    inp = I.w8a8_inputs(cfg, 1, 3, seed=15, positions=[0, 0, 0])
    H, rq = 2, 192
    nq = H * 192
    src = (5 * np.arange(nq) + 1) % rq
    Wqb = np.zeros((rq, nq), dtype=np.int8)
    Wqb[src, np.arange(nq)] = np.where(np.arange(nq) % 3 == 0, -2, 1)
    inp["W_qb"] = torch.from_numpy(Wqb)
    q_nope, q_pe, k_nope, value, k_pe = oracle_mod.w8a8_prolog(inp, nthreads=1)
    for t in range(3):
        q1, s1, c1, s2 = oracle_mod.w8a8_operands(inp, t)
        y = Wqb[src, np.arange(nq)].astype(np.float64) * q1[src] * s1 * inp["s_qb"].numpy()
        for hh in range(H):
            np.testing.assert_allclose(q_nope[0, hh, t], y[hh * 192:hh * 192 + 128], rtol=1e-12)
            pe = y[hh * 192 + 128:hh * 192 + 192]
            # position 0: RoPE is the de-interleave
            np.testing.assert_allclose(q_pe[0, hh, t], np.concatenate([pe[0::2], pe[1::2]]),
                                       rtol=1e-12)


def test_w8a8_first_gemm_is_integer_exact(oracle_mod):
    """The kv_a output equals int_gemm(quant(hidden)) * s_x * s_w: checked
    through k_pe at position 0 (the de-interleaved dequantised columns)."""
    cfg = _tiny_w8_cfg()
    inp = I.w8a8_inputs(cfg, 2, 1, seed=16, positions=[0, 0])
    *_, k_pe = oracle_mod.w8a8_prolog(inp, nthreads=1)
    for t in range(2):
        x = inp["hidden"][t].float().numpy()
        q, sx = oracle_mod.quant_row_f32(x)
        acc = q.astype(np.int64) @ inp["W_kva"].numpy().astype(np.int64)
        y = acc[512:576] * np.float64(sx) * inp["s_kva"].numpy()[512:576].astype(np.float64)
        np.testing.assert_allclose(k_pe[t, 0, 0], np.concatenate([y[0::2], y[1::2]]), rtol=1e-13)


def _w8_routing_case(positions):
    """Closed-form W8A8 case: hidden rows v_t * sign (quantised to +-127
    exactly), one-hot W_qa / W_kva (every latent column of a token has the
    same magnitude, so both RMSNorms are known in closed form), constant
    scales on the normalised columns, and one-hot W_qb / W_kvb."""
    cfg = I.small_config(I.R1_W8A8, hidden=256, q_lora_rank=192, num_heads=2, max_pos=64)
    T, h, rq, r, H = len(positions), 256, 192, 512, 2
    nq, nkv = H * 192, H * 256
    sign = np.where(np.arange(h) % 3 == 1, -1.0, 1.0)
    v = np.array([0.75, 1.5, 3.0, 0.5])[:T]
    hid = v[:, None] * sign[None, :]

    def onehot(K, N, src, w):
        W = np.zeros((K, N), dtype=np.int8)
        W[src, np.arange(N)] = w
        return W

    src_qa = (3 * np.arange(rq) + 1) % h
    w_qa = np.where(np.arange(rq) % 4 == 0, -1, 1)
    src_kva = (5 * np.arange(r + 64) + 2) % h
    w_kva = np.concatenate([np.where(np.arange(r) % 7 == 0, -1, 1), (np.arange(64) % 5) - 2])
    src_qb = (7 * np.arange(nq) + 5) % rq
    w_qb = np.where(np.arange(nq) % 3 == 0, -2, 1)
    src_kvb = (11 * np.arange(nkv) + 3) % r
    w_kvb = np.where(np.arange(nkv) % 5 == 0, 1, -1)
    s_qa = np.full(rq, 0.01, dtype=np.float32)
    s_kva = np.concatenate([np.full(r, 0.02), 0.01 * (1 + np.arange(64) / 64)]).astype(np.float32)
    s_qb = (0.005 + 0.0001 * np.arange(nq)).astype(np.float32)
    s_kvb = (0.004 + 0.0001 * (np.arange(nkv) % 97)).astype(np.float32)
    gq = np.array([0.5, 2.0, 1.0, 1.5])[np.arange(rq) % 4]
    gk = np.array([1.25, 0.75, 2.0])[np.arange(r) % 3]
    cos, sin = I.rope_tables(64, 64, 10000.0)
    bf = torch.bfloat16
    inp = dict(cfg=cfg, b=1, s=T, hidden=torch.tensor(hid).to(bf),
               positions=torch.tensor(positions, dtype=torch.int32), cos=cos, sin=sin,
               W_qa=torch.from_numpy(onehot(h, rq, src_qa, w_qa)), s_qa=torch.from_numpy(s_qa),
               gamma_q=torch.tensor(gq).to(bf),
               W_qb=torch.from_numpy(onehot(rq, nq, src_qb, w_qb)), s_qb=torch.from_numpy(s_qb),
               W_kva=torch.from_numpy(onehot(h, r + 64, src_kva, w_kva)), s_kva=torch.from_numpy(s_kva),
               gamma_kv=torch.tensor(gk).to(bf),
               W_kvb=torch.from_numpy(onehot(r, nkv, src_kvb, w_kvb)), s_kvb=torch.from_numpy(s_kvb))
    return inp, dict(v=v, sign=sign, src_qa=src_qa, w_qa=w_qa, src_kva=src_kva, w_kva=w_kva,
                     src_qb=src_qb, w_qb=w_qb, src_kvb=src_kvb, w_kvb=w_kvb, s_qa=s_qa, s_kva=s_kva,
                     s_qb=s_qb, s_kvb=s_kvb, gq=gq, gk=gk, cos=cos.numpy(), sin=sin.numpy())


def test_w8a8_routing_closed_form(oracle_mod):
    """Every W8A8 output in closed form, at positions 0, 7 and 63.  A row
    v * sign quantises to 127 * sign with scale fp32(v / 127); the one-hot
    q_a / kv_a GEMMs then give latent columns of one magnitude c per token,
    so RMSNorm is sign * c / sqrt(c^2 + eps) * gamma; the requantised
    operands are the (hand-pinned) fp32 quantisation of those vectors; the
    one-hot q_b / kv_b pick w * operand[src] * scale * s_w[j]; q_pe and
    k_pe are the (hand-pinned) RoPE of their columns at the token's
    position.  This pins the Q-side and KV-side norms separately (gamma_q
    vs gamma_kv), both requantisations, the head pitches (192 for q, 256
    for kv), the value columns and the positions."""
    positions = [0, 7, 63]
    inp, k = _w8_routing_case(positions)
    q_nope, q_pe, k_nope, value, k_pe = oracle_mod.w8a8_prolog(inp, nthreads=1)
    eps = 1e-6
    for t, p in enumerate(positions):
        s_x = np.float32(np.float32(k["v"][t]) / np.float32(127))
        # q_a / kv_a: acc = 127 * sign[src] * w, dequantised with s_x * s_w
        yq = 127.0 * k["sign"][k["src_qa"]] * k["w_qa"] * np.float64(s_x) * k["s_qa"].astype(np.float64)
        ya = 127.0 * k["sign"][k["src_kva"]] * k["w_kva"] * np.float64(s_x) * k["s_kva"].astype(np.float64)
        cq = abs(yq[0])
        ck = abs(ya[0])
        nq = np.sign(yq) * cq / math.sqrt(cq * cq + eps) * k["gq"]
        nk = np.sign(ya[:512]) * ck / math.sqrt(ck * ck + eps) * k["gk"]
        q1, s1 = oracle_mod.quant_row_f32(nq.astype(np.float32))
        c1, s2 = oracle_mod.quant_row_f32(nk.astype(np.float32))
        o_q1, o_s1, o_c1, o_s2 = oracle_mod.w8a8_operands(inp, t)
        assert np.array_equal(o_q1, q1) and o_s1 == s1
        assert np.array_equal(o_c1, c1) and o_s2 == s2
        yqb = k["w_qb"] * q1[k["src_qb"]].astype(np.float64) * np.float64(s1) * k["s_qb"].astype(np.float64)
        ykvb = k["w_kvb"] * c1[k["src_kvb"]].astype(np.float64) * np.float64(s2) * k["s_kvb"].astype(np.float64)
        for hh in range(2):
            np.testing.assert_allclose(q_nope[0, hh, t], yqb[hh * 192:hh * 192 + 128], rtol=1e-12)
            np.testing.assert_allclose(q_pe[0, hh, t],
                                       oracle_mod.rope(yqb[hh * 192 + 128:hh * 192 + 192], k["cos"][p],
                                                       k["sin"][p]), rtol=1e-12, atol=1e-15)
            np.testing.assert_allclose(k_nope[0, hh, t], ykvb[hh * 256:hh * 256 + 128], rtol=1e-12)
            np.testing.assert_allclose(value[0, hh, t], ykvb[hh * 256 + 128:hh * 256 + 256], rtol=1e-12)
        np.testing.assert_allclose(k_pe[0, 0, t], oracle_mod.rope(ya[512:576], k["cos"][p], k["sin"][p]),
                                   rtol=1e-12, atol=1e-15)
    # the RoPE is not the identity at these positions
    assert not np.allclose(q_pe[0, 0, 1], q_pe[0, 0, 0])
