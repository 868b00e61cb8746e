"""The pins hold the oracle to the mathematics: each of these planted
mistakes, compiled into a copy of oracle.c, makes the pin suite fail
(the mutant library is loaded through MLA_ORACLE_SO in a child pytest).
The mistakes cover the KV prolog, the latent-cache variant and the W8A8
path (integer GEMM, dequantisation scales, both norms, requantisation,
head pitches, RoPE positions)."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "rotate_half sign": ("double rot = (i < half) ? -xd[i + half] : xd[i - half];",
                         "double rot = (i < half) ? xd[i + half] : xd[i - half];"),
    "eps outside the sqrt": ("double denom = sqrt(ss / (double)n + eps);",
                             "double denom = sqrt(ss / (double)n) + eps;"),
    "dropped K term": ("for (int64_t k = 0; k < K; ++k) acc += x[k] * W[k * N + n];",
                       "for (int64_t k = 1; k < K; ++k) acc += x[k] * W[k * N + n];"),
    "value from the k_nope columns": ("value[hh * d->vdim + i] = KV[hh * hd + d->nope + i];",
                                      "value[hh * d->vdim + i] = KV[hh * hd + i];"),
    "k_pe slice off by one": ("const double* kpe = C + r;", "const double* kpe = C + r + 1;"),
    "no de-interleave": ("xd[j] = x[2 * j];\n    xd[half + j] = x[2 * j + 1];",
                         "xd[j] = x[j];\n    xd[half + j] = x[half + j];"),
    "quantisation truncates": ("float r = rintf(y);", "float r = truncf(y);"),
    "KV RoPE at position 0": (
        "oracle_kv_prolog_token(d, x, Wa, g, Wb, cosb + (int64_t)p * dr, sinb + (int64_t)p * dr, kn,",
        "oracle_kv_prolog_token(d, x, Wa, g, Wb, cosb, sinb, kn,"),
    "latent without RMSNorm": ("oracle_rmsnorm(C, r, g, d->eps, latent + t * r);",
                               "memcpy(latent + t * r, C, sizeof(double) * r);"),
    # W8A8 path (the pin configurations keep q_lora_rank <= kv_lora_rank, so
    # the gamma mix-up below stays inside the gamma_kv buffer)
    "W8A8 int GEMM reads W transposed": (
        "for (int64_t k = 0; k < K; ++k) a += (int64_t)q[k] * (int64_t)W[k * N + n];",
        "for (int64_t k = 0; k < K; ++k) a += (int64_t)q[k] * (int64_t)W[n * K + k];"),
    "W8A8 q heads at the kv head pitch": ("q_nope[hh * d->nope + i] = yb[hh * qhd + i];",
                                          "q_nope[hh * d->nope + i] = yb[hh * kvhd + i];"),
    "W8A8 kv_b dequantised with the q operand scale": (
        "yb[j] = (double)acc_q[j] * (double)s2 * (double)s_kvb[j];",
        "yb[j] = (double)acc_q[j] * (double)s1 * (double)s_kvb[j];"),
    "W8A8 value from the k_nope columns": ("value[hh * d->vdim + i] = yb[hh * kvhd + d->nope + i];",
                                           "value[hh * d->vdim + i] = yb[hh * kvhd + i];"),
    "W8A8 RoPE at position 0": (
        "const float* crow = cosb + (int64_t)p * dr;\n  const float* srow = sinb + (int64_t)p * dr;",
        "const float* crow = cosb;\n  const float* srow = sinb;"),
    "W8A8 k_pe without the activation scale": (
        "ya[n] = (double)acc_a[n] * (double)s_x * (double)s_kva[n];",
        "ya[n] = (double)acc_a[n] * (double)s_kva[n];"),
    "W8A8 activation scale inverted": ("volatile float sc = amax / 127.0f;",
                                       "volatile float sc = 127.0f / amax;"),
    "W8A8 q norm with gamma_kv": ("oracle_rmsnorm(yq, rq, gq, d->eps, nq_);",
                                  "oracle_rmsnorm(yq, rq, gk, d->eps, nq_);"),
    "W8A8 q operand quantised before the norm": (
        "for (int64_t c = 0; c < rq; ++c) nqf[c] = (float)nq_[c];",
        "for (int64_t c = 0; c < rq; ++c) nqf[c] = (float)yq[c];"),
}


def run_pins(src_text, tmp_path):
    """Compile src_text as the oracle and run the pin suite on it in a child pytest."""
    c = tmp_path / "oracle_variant.c"
    c.write_text(src_text)
    so = tmp_path / "liboracle_variant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-shared", "-fPIC",
                    str(c), "-lm", "-o", str(so)], check=True, capture_output=True)
    env = dict(os.environ, MLA_ORACLE_SO=str(so))
    return subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                           os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                          env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)


def test_unmutated_copy_passes(tmp_path):
    r = run_pins(open(SRC).read(), tmp_path)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_the_pins(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    r = run_pins(src.replace(old, new), tmp_path)
    # a pin assertion failed (not a collection or import error)
    assert r.returncode == 1 and " failed" in r.stdout, f"{name}: the pins did not catch it\n{r.stdout[-2000:]}"


# Mistakes in the oracle's Python part (int8 KV-cache codes, paged layout):
# the pin suite runs from a temporary tree holding a mutated copy of the
# oracle package (its C library prebuilt, passed through MLA_ORACLE_SO).
PY_SRC = os.path.join(ROOT, "oracle", "__init__.py")
PY_MUTANTS = {
    "int8 code without the dtype rounding": (
        "xd = round_to(np.nan_to_num(x, nan=0.0), dtype).astype(np.float32)",
        "xd = np.nan_to_num(x, nan=0.0).astype(np.float32)"),
    "int8 code clamped at -128": ("return np.clip(np.rint(y), -127, 127).astype(np.int8)",
                                  "return np.clip(np.rint(y), -128, 127).astype(np.int8)"),
    "int8 code truncates": ("return np.clip(np.rint(y), -127, 127).astype(np.int8)",
                            "return np.clip(np.trunc(y), -127, 127).astype(np.int8)"),
    "paged slot split swapped": ("blk, off = divmod(int(slots[t]), page_size)",
                                 "off, blk = divmod(int(slots[t]), page_size)"),
    "paged negative slot not dropped": ("            if slots[t] < 0:\n                continue\n", ""),
    "paged row from the wrong sequence": ("bi, si = divmod(t, s)\n            c[blk",
                                          "si, bi = divmod(t, b)\n            c[blk"),
}


def run_pins_py(py_text, tmp_path):
    """Run the pin suite against a copy of the oracle package whose Python
    part is py_text."""
    import oracle
    so = oracle.build()
    (tmp_path / "oracle").mkdir()
    (tmp_path / "oracle" / "__init__.py").write_text(py_text)
    shutil.copy(SRC, tmp_path / "oracle")
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), tmp_path / "tests" / "golden")
    for f in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), tmp_path / "tests")
    shutil.copy(os.path.join(ROOT, "pytest.ini"), tmp_path)
    os.symlink(os.path.join(ROOT, "mla_attention_kv_gb300"), tmp_path / "mla_attention_kv_gb300")
    env = dict(os.environ, MLA_ORACLE_SO=so)
    return subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                           str(tmp_path / "tests" / "test_oracle_pins.py")],
                          env=env, cwd=tmp_path, capture_output=True, text=True, timeout=600)


def test_unmutated_python_copy_passes(tmp_path):
    r = run_pins_py(open(PY_SRC).read(), tmp_path)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_planted_python_mistake_fails_the_pins(name, tmp_path):
    old, new = PY_MUTANTS[name]
    src = open(PY_SRC).read()
    assert src.count(old) == 1, name
    r = run_pins_py(src.replace(old, new), tmp_path)
    assert r.returncode == 1 and " failed" in r.stdout, f"{name}: the pins did not catch it\n{r.stdout[-2000:]}"
