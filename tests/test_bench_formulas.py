"""The algorithmic bytes and FLOPs behind bench.py's roofline fractions,
checked against sums written out from the shapes (no GPU: only the
workload descriptions are built).  Per call: every weight byte once, and per
token its hidden row, position, cos/sin rows and outputs; FLOPs are the two
(or four) contractions."""
import pytest

import bench


def test_decode_sweep_points_and_bytes():
    wl = bench.WORKLOADS["decode_sweep"]()
    assert wl.points == [(b, s) for s in (1, 2) for b in (1, 2, 4, 8, 16, 32, 64, 128)]
    assert wl.tokens_per_step == 255 + 510
    # V2-Lite: W_kva 2048 x 576, gamma 512, W_kvb 512 x 4096, fp16
    w = 2 * (2048 * 576 + 512 + 512 * 4096)
    assert wl.weight_bytes() == w == 6_554_624
    # per token: hidden 4096 B, position 4 B, cos + sin rows 512 B, k_nope + value 16 heads x 512 B, k_pe 128 B
    assert wl.alg_bytes(1) == w + 4096 + 4 + 512 + 16 * 512 + 128 == 6_567_556
    assert wl.flops(1) == 2 * (2048 * 576 + 512 * 4096) == 6_553_600


def test_single_call_workloads():
    r1p = bench.WORKLOADS["r1_prefill"]()
    assert r1p.T == 16384
    assert r1p.flops(1) == 2 * (7168 * 576 + 512 * 128 * 256) == 41_811_968
    v2p = bench.WORKLOADS["v2lite_prefill"]()
    assert v2p.flops(16384) == pytest.approx(16384 * 6_553_600)
    r1d = bench.WORKLOADS["r1_decode"]()
    w = 2 * (7168 * 576 + 512 + 512 * 128 * 256)
    assert r1d.alg_bytes(64) == w + 64 * (2 * 7168 + 4 + 512 + 2 * (128 * 256 + 64))


def test_w8a8_bytes():
    wl = bench.WORKLOADS["w8a8_t1"]()
    h, rq, H = 7168, 1536, 128
    weights = h * (rq + 576) + rq * H * 192 + 512 * H * 256          # int8
    scales = 4 * (rq + 576 + H * 192 + H * 256)                      # fp32 per output channel
    gammas = 2 * (rq + 512)                                          # bf16
    per_tok = 2 * h + 4 + 512 + 2 * (H * 256 + 64) + 2 * H * 192     # + q_nope / q_pe outputs
    assert wl.alg_bytes(1) == weights + scales + gammas + per_tok == 70_036_356
    assert wl.flops(1) == 2 * (h * (rq + 576) + rq * H * 192 + 512 * H * 256)


def test_variant_workloads():
    lat = bench.WORKLOADS["r1_latent_prefill"]()
    assert lat.flops(1) == 2 * 7168 * 576
    assert lat.alg_bytes(1) == 2 * (7168 * 576 + 512) + 2 * 7168 + 4 + 512 + 2 * (512 + 64)
    paged = bench.WORKLOADS["r1_paged_prefill"]()
    dense = bench.WORKLOADS["r1_prefill"]()
    assert paged.alg_bytes(16384) == dense.alg_bytes(16384) and paged.flops(1) == dense.flops(1)
    c8 = bench.WORKLOADS["r1_c8_prefill"]()
    T = 16384
    # int8 codes instead of 2-byte values, plus the per-channel scales once
    assert c8.alg_bytes(T) == pytest.approx(
        2 * (7168 * 576 + 512 + 512 * 128 * 256) + T * (2 * 7168 + 4 + 512 + 128 * 256 + 64)
        + 4 * (128 * 256 + 64))
    for name in ("v2lite_latent_decode", "v2lite_paged_decode", "v2lite_c8_decode"):
        d = bench.WORKLOADS[name]().describe()
        assert "variant" in d and d["T"] == 64


@pytest.mark.parametrize("name", sorted(bench.WORKLOADS))
def test_every_workload_describes_itself(name):
    """Each workload names itself and its model with its sizes, serialises
    as the JSON line's config, and has positive work per call."""
    import json
    wl = bench.WORKLOADS[name]()
    d = wl.describe()
    json.dumps(d)
    assert d["workload"] and d["model"]
    assert any(str(x) in d["workload"] for x in ("s2", "s1", "s4096", "s8192", "T1", "T64", "T8192", "sweep"))
    for b, s in wl.points:
        assert wl.alg_bytes(b * s) > wl.weight_bytes() > 0 and wl.flops(b * s) > 0
    assert wl.tokens_per_step == sum(b * s for b, s in wl.points)
