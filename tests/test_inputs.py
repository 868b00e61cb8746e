"""The seeded input generators shared by the oracle tests, the GPU parity
tests and the benchmark: deterministic per seed, the shapes and dtypes of
the ABI, the value distributions and position rules stated in the module
docstring, and the W8A8 weight encoding (no method arithmetic is tested
here)."""
import math

import pytest
import torch

from mla_attention_kv_gb300 import inputs as I


def test_same_seed_same_data_other_seed_other_data():
    cfg = I.small_config(I.V2_LITE, hidden=256, num_heads=2)
    a = I.kv_inputs(cfg, 2, 3, seed=5)
    b = I.kv_inputs(cfg, 2, 3, seed=5)
    c = I.kv_inputs(cfg, 2, 3, seed=6)
    for k in ("hidden", "W_kva", "gamma_kv", "W_kvb", "positions"):
        assert torch.equal(a[k], b[k]), k
    assert not torch.equal(a["hidden"], c["hidden"])


@pytest.mark.parametrize("base", [I.V2_LITE, I.R1])
def test_kv_shapes_and_dtypes(base):
    cfg = I.small_config(base, hidden=128, num_heads=3)
    d = I.kv_inputs(cfg, 2, 5, seed=1)
    dt = torch.float16 if cfg["dtype"] == "fp16" else torch.bfloat16
    assert d["hidden"].shape == (10, 128) and d["hidden"].dtype == dt
    assert d["W_kva"].shape == (128, 576) and d["W_kva"].dtype == dt
    assert d["gamma_kv"].shape == (512,) and d["W_kvb"].shape == (512, 3 * 256)
    assert d["positions"].shape == (10,) and d["positions"].dtype == torch.int32
    assert d["cos"].shape == (cfg["max_pos"], 64) and d["cos"].dtype == torch.float32


def test_value_distributions():
    cfg = I.small_config(I.V2_LITE, hidden=2048, num_heads=4)
    d = I.kv_inputs(cfg, 16, 4, seed=3)
    h = d["hidden"].float()
    assert abs(h.mean().item()) < 0.02 and abs(h.std().item() - 1.0) < 0.02
    for k in ("W_kva", "W_kvb"):
        w = d[k].float()
        assert abs(w.mean().item()) < 1e-3 and abs(w.std().item() - 0.02) < 1e-3, k
    g = d["gamma_kv"].float()
    assert abs(g.mean().item() - 1.0) < 0.02 and abs(g.std().item() - 0.1) < 0.02


def test_positions():
    g = torch.Generator().manual_seed(0)
    pre = I.make_positions(3, 5, "prefill", 4096, g)
    assert pre.tolist() == list(range(5)) * 3
    dec = I.make_positions(64, 2, "decode", 4096, g).view(64, 2)
    assert torch.all(dec[:, 1] == dec[:, 0] + 1)
    assert int(dec.min()) >= 0 and int(dec.max()) <= 4095
    assert len(set(dec[:, 0].tolist())) > 32  # drawn, not constant
    assert I.make_positions(1, 2, [7, 8], 4096, g).tolist() == [7, 8]
    with pytest.raises(ValueError):
        I.make_positions(1, 1, "other", 16, g)


def test_w8a8_weights():
    cfg = I.small_config(I.R1_W8A8, hidden=512, q_lora_rank=256, num_heads=4)
    d = I.w8a8_inputs(cfg, 2, 2, seed=9)
    for w, sc in (("W_qa", "s_qa"), ("W_qb", "s_qb"), ("W_kva", "s_kva"), ("W_kvb", "s_kvb")):
        q, s = d[w], d[sc]
        assert q.dtype == torch.int8 and int(q.min()) >= -127 and int(q.max()) <= 127, w
        assert s.dtype == torch.float32 and s.shape == (q.shape[1],), sc
        assert float(s.min()) >= 0.005 and float(s.max()) <= 0.02, sc
        deq = q.float() * s[None, :]
        # dequantised weights keep the N(0, 0.02) magnitude (within the step s/2)
        assert abs(deq.std().item() - 0.02) < 2e-3, w
    assert d["hidden"].dtype == torch.bfloat16 and d["gamma_q"].shape == (256,)


def test_sampled_rows():
    rows = I.sampled_rows(3, 100, 20, seed=4)
    assert rows == sorted(set(rows))
    assert all(0 <= r < 300 for r in rows)
    for bi in range(3):
        assert bi * 100 in rows and bi * 100 + 99 in rows
    assert len(rows) >= 20


def test_rope_tables():
    cos, sin = I.rope_tables(64, 64, 10000.0)
    assert torch.allclose(cos[:, :32], cos[:, 32:]) and torch.allclose(sin[:, :32], sin[:, 32:])
    assert torch.allclose(cos.double() ** 2 + sin.double() ** 2, torch.ones(64, 64, dtype=torch.float64),
                          atol=1e-6)
    assert cos[0].eq(1).all() and sin[0].eq(0).all()
    # column j at position p is cos(p * theta^(-2j/64)) rounded to fp32
    p, j = 37, 5
    assert cos[p, j].item() == pytest.approx(math.cos(p * 10000.0 ** (-2 * j / 64)), abs=1e-7)


def test_tile_rows_cover_every_tile_and_offset():
    for b, s in ((4, 4096), (2, 8192), (1, 8192), (1, 300), (3, 100)):
        T = b * s
        rows = I.tile_rows(b, s, 512, seed=7)
        assert rows == sorted(set(rows)) and all(0 <= r < T for r in rows)
        assert {r // 128 for r in rows} == set(range((T + 127) // 128))
        if T >= 128:
            assert {r % 128 for r in rows} == set(range(128))
        for bi in range(b):
            assert bi * s in rows and bi * s + s - 1 in rows
        assert len(rows) >= min(T, 512) * 0.8
