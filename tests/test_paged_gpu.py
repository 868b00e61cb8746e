"""GPU checks of the paged KV-cache variant (mla_kv_prolog_run_paged): the
prolog's outputs scattered into block-paged caches by a slot mapping, on
the decode and the prefill kernel.  Written rows must be bit-identical to
the dense run's rows (same arithmetic, different addresses) and within the
parity tolerance of the oracle's scatter; untouched cache entries keep
their contents; negative slots drop rows; slots past the cache drop rows
and are reported."""
import numpy as np
import pytest
import torch

from mla_attention_kv_gb300 import binding as B
from mla_attention_kv_gb300 import build as BLD
from mla_attention_kv_gb300 import inputs as I

from parity import compare

pytestmark = pytest.mark.gpu
NAMES = ("k_cache", "v_cache", "kpe_cache")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    BLD.build()
    B.load()


def make_slots(T, page, nblocks, seed, drop=()):
    """Distinct random slots in [0, nblocks * page); rows in `drop` get -1."""
    g = np.random.default_rng(seed)
    slots = g.permutation(nblocks * page)[:T].astype(np.int32)
    for t in drop:
        slots[t] = -1
    return slots


def run_paged(cfg, b, s, seed, page, nblocks, slots, path, positions="decode", oracle_mod=None,
              rows=None, packed=False):
    inp = I.kv_inputs(cfg, b, s, seed, positions)
    d = B.to_device(inp)
    m = B.MLAProlog(cfg, b * s)
    m.set_path(path)
    if packed:
        m.prepare_weights(d)
    caches = m.alloc_paged_caches(nblocks, page)
    for c in caches.values():
        c.fill_(float("nan"))
    sl = torch.tensor(slots, dtype=torch.int32, device="cuda")
    m.run_paged(b, s, d, sl, page, caches)
    torch.cuda.synchronize()
    st = m.status()
    dense = m.alloc_outputs(b, s)
    m.run(b, s, d, dense)
    torch.cuda.synchronize()
    assert m.status() == 0
    m.close()
    # bit-exact against the dense run, row by row
    H = cfg["num_heads"]
    for t in range(b * s):
        bi, si = divmod(t, s)
        if slots[t] < 0 or slots[t] >= nblocks * page:
            continue
        blk, off = divmod(int(slots[t]), page)
        assert torch.equal(caches["k_cache"][blk, :, off], dense["k_nope"][bi, :, si])
        assert torch.equal(caches["v_cache"][blk, :, off], dense["value"][bi, :, si])
        assert torch.equal(caches["kpe_cache"][blk, 0, off], dense["k_pe"][bi, 0, si])
    # entries no row writes keep their contents (NaN here)
    written = np.zeros((nblocks, page), dtype=bool)
    for t in range(b * s):
        if 0 <= slots[t] < nblocks * page:
            written[divmod(int(slots[t]), page)] = True
    free = torch.tensor(~written, device="cuda")
    for n in NAMES:
        c = caches[n]
        assert torch.all(torch.isnan(c.permute(0, 2, 1, 3)[free])), n
    if oracle_mod is not None:
        ref = oracle_mod.kv_prolog(inp, rows=rows)
        ok = [t for t in range(b * s) if 0 <= slots[t] < nblocks * page]
        paged = oracle_mod.scatter_paged(ref, b, s, np.where(np.isin(np.arange(b * s), ok), slots, -1),
                                         page, nblocks)
        for n, r in zip(NAMES, paged):
            compare(n, caches[n], r, oracle_mod)
    return st


def test_paged_decode_v2lite(oracle_mod):
    b, s, page, nblk = 8, 2, 4, 12
    slots = make_slots(b * s, page, nblk, 1, drop=(3, 10))
    assert run_paged(I.V2_LITE, b, s, 401, page, nblk, slots, B.PATH_DECODE, oracle_mod=oracle_mod) == 0


@pytest.mark.parametrize("packed", [False, True])
def test_paged_decode_r1(oracle_mod, packed):
    # packed R1 weights: kv_b on the tensor cores, the same paged store epilogue
    b, s, page, nblk = 64, 1, 16, 8
    slots = make_slots(b * s, page, nblk, 2)
    assert run_paged(I.R1, b, s, 402, page, nblk, slots, B.PATH_DECODE, oracle_mod=oracle_mod,
                     packed=packed) == 0


def test_paged_decode_two_launches(oracle_mod):
    b, s, page, nblk = 100, 2, 8, 30
    slots = make_slots(b * s, page, nblk, 3, drop=(0, 199))
    assert run_paged(I.V2_LITE, b, s, 403, page, nblk, slots, B.PATH_DECODE, oracle_mod=oracle_mod) == 0


@pytest.mark.parametrize("T", [1024, 1061])
def test_paged_prefill_v2lite(oracle_mod, T):
    page, nblk = 16, (T + 15) // 16 + 3
    slots = make_slots(T, page, nblk, 4, drop=(5, T - 1))
    rows = I.tile_rows(1, T, 512, seed=T)
    assert run_paged(I.V2_LITE, 1, T, 404, page, nblk, slots, B.PATH_PREFILL, positions="prefill",
                     oracle_mod=oracle_mod, rows=rows) == 0


def test_paged_bad_slot_is_reported():
    b, s, page, nblk = 2, 3, 4, 2
    slots = np.array([0, 1, 8, 3, -1, 2], dtype=np.int32)  # slot 8 is past the 8-slot cache
    st = run_paged(I.V2_LITE, b, s, 405, page, nblk, slots, B.PATH_DECODE)
    assert st == 10  # MLA_ERR_BAD_SLOT
