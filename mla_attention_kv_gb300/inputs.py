"""Seeded synthetic inputs for the MLA KV prolog.

This module only draws inputs: shapes, seeds and value distributions.  It
holds none of the prolog's arithmetic, so both the CUDA path and the CPU
oracle can be fed from it.  Everything is drawn on the CPU with a
``torch.Generator`` in float32 and then cast (round-to-nearest-even) to the
I/O dtype, so the device and the oracle see the same bits.

Model dimensions follow "DeepSeek-V2-Lite-Chat MLA KV Prolog 迁移指南",
§精度验证 (hidden 2048, kv_lora_rank 512, rope 64, 16 heads, nope = v = 128,
eps 1e-6) and the DeepSeek-R1 shapes (hidden 7168, 128 heads, q_lora_rank
1536) for the R1 / W8A8 workloads.  The pages publish no tensors, so every
value is synthetic:

* hidden_states ~ N(0, 1); weights ~ N(0, 0.02); RMSNorm gamma = 1 + N(0, 0.1)
* positions: decode -> one start p0 ~ U{0 .. max_pos - s} per sequence and
  positions p0 .. p0+s-1; prefill -> 0 .. s-1 per sequence.
* cos/sin tables [max_pos, 64] (float32): entry [p, i] is cos / sin of
  p * theta^(-2 (i mod 32) / 64), evaluated in float64 and rounded once to
  float32 (theta = 10000).  The tables are inputs of the prolog, shared
  as-is by both sides.
* W8A8: int8 weights q = clamp(rint(w / s_n), -127, 127) from w ~ N(0, 0.02)
  and per-output-channel scales s_n ~ U(0.005, 0.02), so that dequantised
  weights keep the magnitude of the floating-point workloads.
"""
from __future__ import annotations

import torch

V2_LITE = dict(name="v2lite", hidden=2048, kv_lora_rank=512, rope_dim=64, num_heads=16,
               nope_dim=128, v_dim=128, dtype="fp16", eps=1e-6, max_pos=4096, theta=10000.0)
R1 = dict(name="r1", hidden=7168, kv_lora_rank=512, rope_dim=64, num_heads=128, nope_dim=128,
          v_dim=128, dtype="bf16", eps=1e-6, max_pos=32768, theta=10000.0)
R1_W8A8 = dict(R1, name="r1_w8a8", q_lora_rank=1536, quant="w8a8")

CONFIGS = {"v2lite": V2_LITE, "r1": R1, "r1_w8a8": R1_W8A8}


def torch_dtype(cfg) -> torch.dtype:
    return torch.float16 if cfg["dtype"] == "fp16" else torch.bfloat16


def small_config(base: dict, **over) -> dict:
    """A copy of ``base`` with some dimensions replaced (tiny test shapes)."""
    c = dict(base)
    c.update(over)
    c["name"] = base["name"] + "_custom"
    return c


def rope_tables(max_pos: int, dim: int = 64, theta: float = 10000.0):
    """cos, sin tables [max_pos, dim] float32 (see the module docstring)."""
    half = dim // 2
    p = torch.arange(max_pos, dtype=torch.float64)[:, None]
    j = torch.arange(dim, dtype=torch.float64)[None, :] % half
    ang = p * torch.pow(torch.tensor(theta, dtype=torch.float64), -2.0 * j / dim)
    return torch.cos(ang).to(torch.float32).contiguous(), torch.sin(ang).to(torch.float32).contiguous()


def make_positions(b: int, s: int, mode, max_pos: int, gen: torch.Generator) -> torch.Tensor:
    if isinstance(mode, (list, tuple)):
        pos = torch.tensor(list(mode), dtype=torch.int32)
        assert pos.numel() == b * s
        return pos
    if mode == "prefill":
        return torch.arange(s, dtype=torch.int32).repeat(b)
    if mode == "decode":
        p0 = torch.randint(0, max_pos - s + 1, (b,), generator=gen, dtype=torch.int64)
        return (p0[:, None] + torch.arange(s)[None, :]).reshape(-1).to(torch.int32)
    raise ValueError(mode)


_TABLE_CACHE: dict = {}


def _tables(cfg):
    key = (cfg["max_pos"], cfg["rope_dim"], cfg["theta"])
    if key not in _TABLE_CACHE:
        _TABLE_CACHE[key] = rope_tables(*key)
    return _TABLE_CACHE[key]


def kv_inputs(cfg: dict, b: int, s: int, seed: int, positions="decode") -> dict:
    """Inputs of the floating-point KV prolog, on the CPU.

    Tensor order (fixed, so a seed means the same data everywhere): hidden,
    W_kva, gamma_kv, W_kvb, positions."""
    g = torch.Generator().manual_seed(seed)
    dt = torch_dtype(cfg)
    h, r, dr, H = cfg["hidden"], cfg["kv_lora_rank"], cfg["rope_dim"], cfg["num_heads"]
    nb = H * (cfg["nope_dim"] + cfg["v_dim"])
    hidden = torch.randn(b * s, h, generator=g).to(dt)
    W_kva = (torch.randn(h, r + dr, generator=g) * 0.02).to(dt)
    gamma_kv = (1.0 + 0.1 * torch.randn(r, generator=g)).to(dt)
    W_kvb = (torch.randn(r, nb, generator=g) * 0.02).to(dt)
    pos = make_positions(b, s, positions, cfg["max_pos"], g)
    cos, sin = _tables(cfg)
    return dict(cfg=cfg, b=b, s=s, hidden=hidden, W_kva=W_kva, gamma_kv=gamma_kv, W_kvb=W_kvb,
                positions=pos, cos=cos, sin=sin)


def _quant_weight(w: torch.Tensor, scale: torch.Tensor) -> torch.Tensor:
    return torch.clamp(torch.round(w / scale[None, :]), -127, 127).to(torch.int8)


def w8a8_inputs(cfg: dict, b: int, s: int, seed: int, positions="decode") -> dict:
    """Inputs of the W8A8 full prolog (bf16 activations, int8 weights).

    Order: hidden, W_kva, gamma_kv, W_kvb, positions, W_qa, s_qa, gamma_q,
    W_qb, s_qb, s_kva, s_kvb."""
    g = torch.Generator().manual_seed(seed)
    h, r, dr, H = cfg["hidden"], cfg["kv_lora_rank"], cfg["rope_dim"], cfg["num_heads"]
    rq = cfg["q_lora_rank"]
    nkv = H * (cfg["nope_dim"] + cfg["v_dim"])
    nq = H * (cfg["nope_dim"] + dr)
    hidden = torch.randn(b * s, h, generator=g).to(torch.bfloat16)
    w_kva = torch.randn(h, r + dr, generator=g) * 0.02
    gamma_kv = (1.0 + 0.1 * torch.randn(r, generator=g)).to(torch.bfloat16)
    w_kvb = torch.randn(r, nkv, generator=g) * 0.02
    pos = make_positions(b, s, positions, cfg["max_pos"], g)
    w_qa = torch.randn(h, rq, generator=g) * 0.02
    s_qa = torch.rand(rq, generator=g) * 0.015 + 0.005
    gamma_q = (1.0 + 0.1 * torch.randn(rq, generator=g)).to(torch.bfloat16)
    w_qb = torch.randn(rq, nq, generator=g) * 0.02
    s_qb = torch.rand(nq, generator=g) * 0.015 + 0.005
    s_kva = torch.rand(r + dr, generator=g) * 0.015 + 0.005
    s_kvb = torch.rand(nkv, generator=g) * 0.015 + 0.005
    cos, sin = _tables(cfg)
    return dict(cfg=cfg, b=b, s=s, hidden=hidden, positions=pos, cos=cos, sin=sin,
                W_qa=_quant_weight(w_qa, s_qa), s_qa=s_qa.float().contiguous(), gamma_q=gamma_q,
                W_qb=_quant_weight(w_qb, s_qb), s_qb=s_qb.float().contiguous(),
                W_kva=_quant_weight(w_kva, s_kva), s_kva=s_kva.float().contiguous(),
                gamma_kv=gamma_kv,
                W_kvb=_quant_weight(w_kvb, s_kvb), s_kvb=s_kvb.float().contiguous())


def seed_for(config_index: int, point: int | None = None) -> int:
    """Seeds: 1000 + config index; sweep points 1100 + point index."""
    return 1100 + point if point is not None else 1000 + config_index


def sampled_rows(b: int, s: int, n: int, seed: int) -> list:
    """Token rows for sampled parity at full size: the first and last row of
    every sequence plus ``n`` seeded random rows, sorted and unique."""
    g = torch.Generator().manual_seed(seed)
    rows = set()
    for bi in range(b):
        rows.add(bi * s)
        rows.add(bi * s + s - 1)
    T = b * s
    if T > 0:
        rows.update(torch.randint(0, T, (n,), generator=g).tolist())
    return sorted(rows)



def tile_rows(b: int, s: int, n: int, seed: int, tile: int = 128) -> list:
    """Token rows for sampled parity at full size that reach every part of a
    tiled kernel: the first and last row of every sequence, at least one row
    in every ``tile``-row tile and at least one row at every offset 0 ..
    tile-1 within a tile (tiles and offsets paired by a seeded shuffle),
    plus ``n`` seeded random rows; sorted and unique."""
    g = torch.Generator().manual_seed(seed)
    T = b * s
    rows = set(sampled_rows(b, s, n, seed))
    if T == 0:
        return []
    ntiles = (T + tile - 1) // tile
    offs = torch.randperm(tile, generator=g).tolist()
    tiles = torch.randperm(ntiles, generator=g).tolist()
    for i in range(max(ntiles, tile)):
        r = tiles[i % ntiles] * tile + offs[i % tile]
        if r >= T:  # the last tile is ragged: any row of it
            r = tiles[i % ntiles] * tile + offs[i % tile] % (T - tiles[i % ntiles] * tile)
        rows.add(r)
    return sorted(rows)
