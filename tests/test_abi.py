"""C-ABI library: builds, loads, exports every declared symbol, and rejects
bad arguments on the host (no GPU needed for any of these)."""
import ctypes
import os
import re

import pytest

from mla_attention_kv_gb300 import binding as B
from mla_attention_kv_gb300 import build as BLD

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    BLD.build()
    return B.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mla_prolog.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_binding_surface():
    assert set(declared_functions()) == set(B.EXPORTED)


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_abi_version_and_strings(L):
    assert L.mla_abi_version() == 1
    for code in range(11):
        assert L.mla_status_string(code).decode() not in ("", "unknown status")
    assert L.mla_status_string(99).decode() == "unknown status"


def _cfg(**over):
    c = dict(hidden=2048, kv_lora_rank=512, rope_dim=64, num_heads=16, nope_dim=128, v_dim=128,
             dtype=B.MLA_F16, eps=1e-6, max_tokens=16, max_pos=4096, quant=0, q_lora_rank=0,
             spin_budget_ns=0)
    c.update(over)
    return B.Config(**c)


@pytest.mark.parametrize("over,code", [
    (dict(hidden=0), 1), (dict(num_heads=0), 1), (dict(max_tokens=0), 1), (dict(max_pos=0), 1),
    (dict(eps=-1.0), 1), (dict(dtype=5), 1), (dict(quant=3), 1),
    (dict(kv_lora_rank=256), 2), (dict(rope_dim=32), 2), (dict(nope_dim=64), 2),
    (dict(v_dim=64), 2), (dict(hidden=2000), 2),
    (dict(quant=1, dtype=B.MLA_F16, q_lora_rank=1536), 2),
    (dict(quant=1, dtype=B.MLA_BF16, q_lora_rank=100), 2),
])
def test_create_rejects_bad_config(L, over, code):
    h = ctypes.c_void_p()
    assert L.mla_kv_prolog_create(ctypes.byref(_cfg(**over)), ctypes.byref(h)) == code
    assert not h.value


def test_null_arguments(L):
    h = ctypes.c_void_p()
    assert L.mla_kv_prolog_create(None, ctypes.byref(h)) == 1
    assert L.mla_kv_prolog_run(None, 1, 1, *([None] * 10), None) == 1
    assert L.mla_prolog_w8a8_run(None, 1, 1, *([None] * 19), None) == 1
    assert L.mla_kv_prolog_status(None, None) == 1
    assert L.mla_kv_prolog_destroy(None) == 1
    assert L.mla_kv_prolog_set_path(None, 0) == 1
    assert L.mla_kv_prolog_last_launches(None) == -1
    assert L.mla_kv_prolog_last_cluster_launches(None) == -1
    assert L.mla_prolog_w8a8_operands(None, 1, None, None, None, None, None) == 1
    assert L.mla_kv_prolog_auto_threshold(None) == -1
    assert L.mla_prolog_w8a8_capture(None, None, None, None) == 1


def test_building_block_shape_checks(L):
    # K must be a multiple of 32 and N of 8 for the int8 GEMM; zero rows is a no-op
    assert L.mla_w8a8_gemm_s32(None, None, 4, 48, 64, None, None) == 2
    assert L.mla_w8a8_gemm_s32(None, None, 4, 64, 96, None, None) == 2
    assert L.mla_w8a8_gemm_s32(None, None, 0, 64, 64, None, None) == 0
    assert L.mla_w8a8_gemm_s32(None, None, 4, 64, 64, None, None) == 1
    assert L.mla_w8a8_quant_rows(None, 4, 12, None, None, None) == 2
    assert L.mla_w8a8_quant_rows(None, 0, 16, None, None, None) == 0
    assert L.mla_w8a8_quant_rows(None, -1, 16, None, None, None) == 1


def test_variant_entries_reject_bad_arguments(L):
    """The latent, paged and int8-cache entries check their own arguments
    before touching the handle or the device."""
    P = ctypes.c_void_p
    fake = P(16)  # never dereferenced: every call below fails its argument check first
    # latent: a null latent output
    assert L.mla_kv_prolog_run_latent(None, 1, 1, *([None] * 8), None) == 1
    # paged: null slot mapping, non-positive page size or block count, slot-count overflow
    args = [fake] * 7
    assert L.mla_kv_prolog_run_paged(fake, 1, 1, *args, None, 16, 4, fake, fake, fake, None) == 1
    assert L.mla_kv_prolog_run_paged(fake, 1, 1, *args, fake, 0, 4, fake, fake, fake, None) == 1
    assert L.mla_kv_prolog_run_paged(fake, 1, 1, *args, fake, 16, 0, fake, fake, fake, None) == 1
    assert L.mla_kv_prolog_run_paged(fake, 1, 1, *args, fake, 1 << 16, 1 << 16, fake, fake, fake, None) == 1
    # paged: a slot mapping that is not 16-byte aligned
    assert L.mla_kv_prolog_run_paged(fake, 1, 1, *args, P(20), 16, 4, fake, fake, fake, None) == 4
    # int8 cache: null or misaligned scale vectors
    assert L.mla_kv_prolog_run_c8(fake, 1, 1, *([fake] * 7), None, fake, fake, fake, fake, fake, None) == 1
    assert L.mla_kv_prolog_run_c8(fake, 1, 1, *([fake] * 7), P(20), fake, fake, fake, fake, fake, None) == 4
    assert B.STATUS_NAMES[10] == "MLA_ERR_BAD_SLOT"
    assert b"slot" in L.mla_status_string(10)


def header_prototypes():
    """{name: [kind of each parameter]} from include/mla_prolog.h, kinds
    'ptr' (pointers, handles, streams), 'int', 'float'."""
    src = open(os.path.join(ROOT, "include", "mla_prolog.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    protos = {}
    for m in re.finditer(r"\b(?:mla_status|int|const char\s*\*)\s+(mla_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", src):
        params = [p.strip() for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
        kinds = []
        for p in params:
            if "*" in p or "cudaStream_t" in p or "mla_prolog_t" in p:
                kinds.append("ptr")
            elif re.match(r"(const\s+)?float\b", p):
                kinds.append("float")
            else:
                kinds.append("int")
        protos[m.group(1)] = kinds
    return protos


def test_binding_argtypes_match_the_header(L):
    """Every declared function is bound with the header's parameter count,
    and pointer / integer parameters in the same places."""
    protos = header_prototypes()
    assert set(protos) == set(declared_functions())
    src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "mla_prolog.h")).read(), flags=re.S)
    for name in protos:
        ret = re.search(r"(mla_status|int|const char\s*\*)\s+" + name + r"\s*\(", src).group(1)
        want = ctypes.c_char_p if ret.startswith("const char") else ctypes.c_int
        assert getattr(L, name).restype is want, (name, ret)
    for name, kinds in protos.items():
        at = getattr(L, name).argtypes
        if at is None:  # bound without argtypes: only zero-parameter functions
            assert kinds == [], name
            continue
        assert len(at) == len(kinds), (name, len(at), len(kinds))
        for i, (t, k) in enumerate(zip(at, kinds)):
            is_ptr = t is ctypes.c_void_p or t is ctypes.c_char_p or hasattr(t, "_type_") and t.__name__.startswith("LP_")
            if k == "ptr":
                assert is_ptr, (name, i, t)
            elif k == "int":
                assert t is ctypes.c_int, (name, i, t)
            else:
                assert t is ctypes.c_float, (name, i, t)


def test_config_struct_layout_matches_the_header(tmp_path):
    """binding.Config has the header's fields in order with the same types,
    and the same size and field offsets as the C compiler gives the struct."""
    import shutil
    import subprocess
    src = open(os.path.join(ROOT, "include", "mla_prolog.h")).read()
    body = re.search(r"typedef struct mla_prolog_config \{(.*?)\} mla_prolog_config;", src, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = [re.match(r"\s*(.*?)\s+(\w+)$", f.strip()).groups() for f in body.split(";") if f.strip()]
    ctypes_of = {"int": ctypes.c_int, "float": ctypes.c_float, "unsigned long long": ctypes.c_ulonglong}
    assert [(n, ctypes_of[t]) for t, n in fields] == list(B.Config._fields_)
    gcc = shutil.which("gcc")
    cuda_inc = "/usr/local/cuda/include"
    if gcc is None or not os.path.isdir(cuda_inc):
        pytest.skip("gcc or the CUDA headers are missing")
    prog = tmp_path / "layout.c"
    prog.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "mla_prolog.h"\nint main(void) {\n'
                    '  printf("%zu\\n", sizeof(mla_prolog_config));\n'
                    + "".join(f'  printf("%zu\\n", offsetof(mla_prolog_config, {n}));\n' for _, n in fields)
                    + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([gcc, str(prog), "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, "-o", str(exe)],
                   check=True, capture_output=True)
    out = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert out[0] == ctypes.sizeof(B.Config)
    assert out[1:] == [getattr(B.Config, n).offset for _, n in fields]


def test_enum_values_match_the_header():
    src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "mla_prolog.h")).read(), flags=re.S)
    enums = {n: int(v) for n, v in re.findall(r"\b(MLA_[A-Z0-9_]+)\s*=\s*(\d+)", src)}
    assert {v: k for k, v in enums.items() if k.startswith(("MLA_OK", "MLA_ERR_"))} == B.STATUS_NAMES
    assert (enums["MLA_F16"], enums["MLA_BF16"]) == (B.MLA_F16, B.MLA_BF16)
    assert (enums["MLA_QUANT_NONE"], enums["MLA_QUANT_W8A8"]) == (B.QUANT_NONE, B.QUANT_W8A8)
    assert (enums["MLA_PATH_AUTO"], enums["MLA_PATH_DECODE"], enums["MLA_PATH_PREFILL"],
            enums["MLA_PATH_DECODE_GRID"]) == (B.PATH_AUTO, B.PATH_DECODE, B.PATH_PREFILL, B.PATH_DECODE_GRID)


def test_noalloc_rejects_bad_arguments_on_the_host(L):
    """mla_kv_prolog_run_noalloc validates before any CUDA call: no config,
    negative sizes, a W8A8 config, unsupported dimensions, null and
    misaligned pointers; T = 0 is a no-op.  (Fake addresses: nothing is
    dereferenced on these paths.)"""
    good = [ctypes.c_void_p(0x10000 + 0x1000 * i) for i in range(10)]
    status = ctypes.c_void_p(0x90000)
    run = L.mla_kv_prolog_run_noalloc
    assert run(None, 1, 1, *good, status, None) == 1
    assert run(ctypes.byref(_cfg()), -1, 1, *good, status, None) == 1
    assert run(ctypes.byref(_cfg(dtype=7)), 1, 1, *good, status, None) == 1
    assert run(ctypes.byref(_cfg(quant=1, dtype=B.MLA_BF16, q_lora_rank=1536)), 1, 1, *good, status, None) == 9
    assert run(ctypes.byref(_cfg(kv_lora_rank=256)), 1, 1, *good, status, None) == 2
    assert run(ctypes.byref(_cfg(hidden=2000)), 1, 1, *good, status, None) == 2
    assert run(ctypes.byref(_cfg()), 0, 5, *good, status, None) == 0
    for i in range(10):
        args = list(good)
        args[i] = None
        assert run(ctypes.byref(_cfg()), 1, 1, *args, status, None) == 1, i
        args[i] = ctypes.c_void_p(good[i].value + 8)
        assert run(ctypes.byref(_cfg()), 1, 1, *args, status, None) == 4, i
