"""Thin ctypes binding of libmla_prolog.so (include/mla_prolog.h).

Argument marshalling only: every step of the prolog runs in the library's
CUDA kernels.  PyTorch supplies device memory and streams.  There is no CPU
fallback; if the library is missing or the tensors are not on a CUDA
device, the calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

MLA_OK = 0
STATUS_NAMES = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED",
                3: "MLA_ERR_TOO_MANY_TOKENS", 4: "MLA_ERR_MISALIGNED", 5: "MLA_ERR_CUDA",
                6: "MLA_ERR_DEVICE_TIMEOUT", 7: "MLA_ERR_BAD_POSITION", 8: "MLA_ERR_NO_MEMORY",
                9: "MLA_ERR_WRONG_MODE", 10: "MLA_ERR_BAD_SLOT"}
PATH_AUTO, PATH_DECODE, PATH_PREFILL, PATH_DECODE_GRID = 0, 1, 2, 3
MLA_F16, MLA_BF16 = 0, 1
QUANT_NONE, QUANT_W8A8 = 0, 1

EXPORTED = ["mla_kv_prolog_create", "mla_kv_prolog_run", "mla_prolog_w8a8_run",
            "mla_kv_prolog_status", "mla_kv_prolog_destroy", "mla_kv_prolog_set_path",
            "mla_kv_prolog_last_launches", "mla_kv_prolog_last_path", "mla_w8a8_quant_rows",
            "mla_w8a8_gemm_s32", "mla_prolog_w8a8_operands", "mla_status_string",
            "mla_last_cuda_error", "mla_abi_version", "mla_kv_prolog_run_noalloc",
            "mla_kv_prolog_prepare_weights", "mla_kv_prolog_run_latent", "mla_kv_prolog_run_paged",
            "mla_kv_prolog_run_c8", "mla_kv_prolog_auto_threshold", "mla_prolog_w8a8_capture",
            "mla_kv_prolog_last_cluster_launches"]


class MLAError(RuntimeError):
    def __init__(self, code: int, what: str, detail: str = ""):
        self.code = code
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)}" + (f" ({detail})" if detail else ""))


class Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("kv_lora_rank", ctypes.c_int),
                ("rope_dim", ctypes.c_int), ("num_heads", ctypes.c_int),
                ("nope_dim", ctypes.c_int), ("v_dim", ctypes.c_int), ("dtype", ctypes.c_int),
                ("eps", ctypes.c_float), ("max_tokens", ctypes.c_int), ("max_pos", ctypes.c_int),
                ("quant", ctypes.c_int), ("q_lora_rank", ctypes.c_int),
                ("spin_budget_ns", ctypes.c_ulonglong)]


_lib = None


def lib_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load the shared library (built in-tree by build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(path)
    P, I, H = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
    L.mla_kv_prolog_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(ctypes.c_void_p)]
    L.mla_kv_prolog_run.argtypes = [H, I, I] + [P] * 10 + [P]
    L.mla_kv_prolog_run_latent.argtypes = [H, I, I] + [P] * 8 + [P]
    L.mla_kv_prolog_run_paged.argtypes = [H, I, I] + [P] * 8 + [I, I] + [P] * 3 + [P]
    L.mla_kv_prolog_run_c8.argtypes = [H, I, I] + [P] * 13 + [P]
    L.mla_prolog_w8a8_run.argtypes = [H, I, I] + [P] * 19 + [P]
    L.mla_kv_prolog_status.argtypes = [H, P]
    L.mla_kv_prolog_destroy.argtypes = [H]
    L.mla_kv_prolog_set_path.argtypes = [H, I]
    L.mla_kv_prolog_last_launches.argtypes = [H]
    L.mla_kv_prolog_last_path.argtypes = [H]
    L.mla_kv_prolog_last_cluster_launches.argtypes = [H]
    L.mla_w8a8_quant_rows.argtypes = [P, I, I, P, P, P]
    L.mla_w8a8_gemm_s32.argtypes = [P, P, I, I, I, P, P]
    L.mla_prolog_w8a8_operands.argtypes = [H, I, P, P, P, P, P]
    L.mla_kv_prolog_run_noalloc.argtypes = [ctypes.POINTER(Config), I, I] + [P] * 11 + [P]
    L.mla_kv_prolog_prepare_weights.argtypes = [H, P, P, P]
    L.mla_kv_prolog_auto_threshold.argtypes = [H]
    L.mla_prolog_w8a8_capture.argtypes = [H, P, P, P]
    for fn in ("mla_kv_prolog_create", "mla_kv_prolog_run", "mla_prolog_w8a8_run",
               "mla_kv_prolog_status", "mla_kv_prolog_destroy", "mla_kv_prolog_set_path",
               "mla_kv_prolog_last_launches", "mla_kv_prolog_last_path", "mla_w8a8_quant_rows",
               "mla_w8a8_gemm_s32", "mla_prolog_w8a8_operands", "mla_abi_version",
               "mla_kv_prolog_run_noalloc", "mla_kv_prolog_prepare_weights", "mla_kv_prolog_run_latent",
               "mla_kv_prolog_run_paged", "mla_kv_prolog_run_c8", "mla_kv_prolog_auto_threshold",
               "mla_prolog_w8a8_capture", "mla_kv_prolog_last_cluster_launches"):
        getattr(L, fn).restype = ctypes.c_int
    L.mla_status_string.argtypes = [ctypes.c_int]
    L.mla_status_string.restype = ctypes.c_char_p
    L.mla_last_cuda_error.argtypes = []
    L.mla_last_cuda_error.restype = ctypes.c_char_p
    _lib = L
    return L


def _check(code: int, what: str):
    if code != MLA_OK:
        detail = load().mla_last_cuda_error().decode() if code == 5 else ""
        raise MLAError(code, what, detail)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t: torch.Tensor, dtype, name: str) -> int:
    """Device address of a contiguous CUDA tensor of `dtype` (None: any)."""
    # one combined test on the common path (this runs ~10 times per call)
    if isinstance(t, torch.Tensor) and t.is_cuda and (dtype is None or t.dtype is dtype) \
            and t.is_contiguous():
        return t.data_ptr()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    raise ValueError(f"{name} must be contiguous")


def _tdt(cfg: dict) -> torch.dtype:
    return torch.float16 if cfg["dtype"] == "fp16" else torch.bfloat16


# ------------------------------------------------------------------ C-named calls
def _config(cfg: dict, max_tokens: int, spin_budget_ns: int = 0) -> Config:
    return Config(cfg["hidden"], cfg["kv_lora_rank"], cfg["rope_dim"], cfg["num_heads"],
                  cfg["nope_dim"], cfg["v_dim"], MLA_F16 if cfg["dtype"] == "fp16" else MLA_BF16,
                  cfg["eps"], max_tokens, cfg["max_pos"],
                  QUANT_W8A8 if cfg.get("quant") == "w8a8" else QUANT_NONE,
                  cfg.get("q_lora_rank", 0), spin_budget_ns)


def mla_kv_prolog_create(cfg: dict, max_tokens: int, spin_budget_ns: int = 0) -> ctypes.c_void_p:
    c = _config(cfg, max_tokens, spin_budget_ns)
    h = ctypes.c_void_p()
    _check(load().mla_kv_prolog_create(ctypes.byref(c), ctypes.byref(h)), "mla_kv_prolog_create")
    return h


def mla_kv_prolog_destroy(h):
    _check(load().mla_kv_prolog_destroy(h), "mla_kv_prolog_destroy")


def mla_kv_prolog_status(h, stream=None) -> int:
    """Returns the raw status code (0 = ok, 6 = timeout, 7 = bad position)."""
    return load().mla_kv_prolog_status(h, _stream(stream))


def mla_kv_prolog_set_path(h, path: int):
    _check(load().mla_kv_prolog_set_path(h, path), "mla_kv_prolog_set_path")


def mla_kv_prolog_run(h, cfg, b, s, hidden, positions, W_kva, gamma_kv, W_kvb, cos, sin,
                      k_nope, value, k_pe, stream=None):
    dt = _tdt(cfg)
    args = [_dev(hidden, dt, "hidden_states"), _dev(positions, torch.int32, "positions"),
            _dev(W_kva, dt, "W_kva"), _dev(gamma_kv, dt, "gamma_kv"), _dev(W_kvb, dt, "W_kvb"),
            _dev(cos, torch.float32, "cos"), _dev(sin, torch.float32, "sin"),
            _dev(k_nope, dt, "k_nope"), _dev(value, dt, "value"), _dev(k_pe, dt, "k_pe")]
    _check(load().mla_kv_prolog_run(h, b, s, *args, _stream(stream)), "mla_kv_prolog_run")


def mla_kv_prolog_run_latent(h, cfg, b, s, hidden, positions, W_kva, gamma_kv, cos, sin, latent,
                             k_pe, stream=None):
    dt = _tdt(cfg)
    args = [_dev(hidden, dt, "hidden_states"), _dev(positions, torch.int32, "positions"),
            _dev(W_kva, dt, "W_kva"), _dev(gamma_kv, dt, "gamma_kv"),
            _dev(cos, torch.float32, "cos"), _dev(sin, torch.float32, "sin"),
            _dev(latent, dt, "latent"), _dev(k_pe, dt, "k_pe")]
    _check(load().mla_kv_prolog_run_latent(h, b, s, *args, _stream(stream)), "mla_kv_prolog_run_latent")


def mla_kv_prolog_run_paged(h, cfg, b, s, hidden, positions, W_kva, gamma_kv, W_kvb, cos, sin,
                            slot_mapping, page_size, num_blocks, k_cache, v_cache, kpe_cache,
                            stream=None):
    dt = _tdt(cfg)
    args = [_dev(hidden, dt, "hidden_states"), _dev(positions, torch.int32, "positions"),
            _dev(W_kva, dt, "W_kva"), _dev(gamma_kv, dt, "gamma_kv"), _dev(W_kvb, dt, "W_kvb"),
            _dev(cos, torch.float32, "cos"), _dev(sin, torch.float32, "sin"),
            _dev(slot_mapping, torch.int32, "slot_mapping")]
    caches = [_dev(k_cache, dt, "k_cache"), _dev(v_cache, dt, "v_cache"), _dev(kpe_cache, dt, "kpe_cache")]
    _check(load().mla_kv_prolog_run_paged(h, b, s, *args, page_size, num_blocks, *caches, _stream(stream)),
           "mla_kv_prolog_run_paged")


def mla_kv_prolog_run_c8(h, cfg, b, s, hidden, positions, W_kva, gamma_kv, W_kvb, cos, sin,
                         k_scale, v_scale, kpe_scale, k_nope, value, k_pe, stream=None):
    dt, f32, i8 = _tdt(cfg), torch.float32, torch.int8
    args = [_dev(hidden, dt, "hidden_states"), _dev(positions, torch.int32, "positions"),
            _dev(W_kva, dt, "W_kva"), _dev(gamma_kv, dt, "gamma_kv"), _dev(W_kvb, dt, "W_kvb"),
            _dev(cos, f32, "cos"), _dev(sin, f32, "sin"), _dev(k_scale, f32, "k_scale"),
            _dev(v_scale, f32, "v_scale"), _dev(kpe_scale, f32, "kpe_scale"),
            _dev(k_nope, i8, "k_nope"), _dev(value, i8, "value"), _dev(k_pe, i8, "k_pe")]
    _check(load().mla_kv_prolog_run_c8(h, b, s, *args, _stream(stream)), "mla_kv_prolog_run_c8")


def mla_kv_prolog_prepare_weights(h, cfg, W_kva, W_kvb, stream=None):
    """Snapshot W_kva / W_kvb in the decode kernel's packed layout (None, None forgets it)."""
    if W_kva is None and W_kvb is None:
        _check(load().mla_kv_prolog_prepare_weights(h, None, None, _stream(stream)),
               "mla_kv_prolog_prepare_weights")
        return
    dt = _tdt(cfg)
    _check(load().mla_kv_prolog_prepare_weights(h, _dev(W_kva, dt, "W_kva"), _dev(W_kvb, dt, "W_kvb"),
                                                _stream(stream)), "mla_kv_prolog_prepare_weights")


def mla_prolog_w8a8_run(h, b, s, hidden, positions, W_qa, sW_qa, gamma_q, W_qb, sW_qb, W_kva,
                        sW_kva, gamma_kv, W_kvb, sW_kvb, cos, sin, q_nope, q_pe, k_nope, value,
                        k_pe, stream=None):
    bf, i8, f32 = torch.bfloat16, torch.int8, torch.float32
    args = [_dev(hidden, bf, "hidden_states"), _dev(positions, torch.int32, "positions"),
            _dev(W_qa, i8, "W_qa"), _dev(sW_qa, f32, "sW_qa"), _dev(gamma_q, bf, "gamma_q"),
            _dev(W_qb, i8, "W_qb"), _dev(sW_qb, f32, "sW_qb"), _dev(W_kva, i8, "W_kva"),
            _dev(sW_kva, f32, "sW_kva"), _dev(gamma_kv, bf, "gamma_kv"),
            _dev(W_kvb, i8, "W_kvb"), _dev(sW_kvb, f32, "sW_kvb"), _dev(cos, f32, "cos"),
            _dev(sin, f32, "sin"), _dev(q_nope, bf, "q_nope"), _dev(q_pe, bf, "q_pe"),
            _dev(k_nope, bf, "k_nope"), _dev(value, bf, "value"), _dev(k_pe, bf, "k_pe")]
    _check(load().mla_prolog_w8a8_run(h, b, s, *args, _stream(stream)), "mla_prolog_w8a8_run")


def mla_kv_prolog_run_noalloc(cfg, b, s, hidden, positions, W_kva, gamma_kv, W_kvb, cos, sin,
                              k_nope, value, k_pe, device_status=None, stream=None):
    """The allocation-free entry point: same computation as mla_kv_prolog_run,
    no handle, scratch in the library's fixed device array."""
    dt = _tdt(cfg)
    c = _config(cfg, max(1, b * s))
    args = [_dev(hidden, dt, "hidden_states"), _dev(positions, torch.int32, "positions"),
            _dev(W_kva, dt, "W_kva"), _dev(gamma_kv, dt, "gamma_kv"), _dev(W_kvb, dt, "W_kvb"),
            _dev(cos, torch.float32, "cos"), _dev(sin, torch.float32, "sin"),
            _dev(k_nope, dt, "k_nope"), _dev(value, dt, "value"), _dev(k_pe, dt, "k_pe"),
            None if device_status is None else _dev(device_status, torch.int32, "device_status")]
    _check(load().mla_kv_prolog_run_noalloc(ctypes.byref(c), b, s, *args, _stream(stream)),
           "mla_kv_prolog_run_noalloc")


def mla_w8a8_quant_rows(x, q, scale, stream=None):
    rows, cols = x.shape
    _check(load().mla_w8a8_quant_rows(_dev(x, torch.bfloat16, "x"), rows, cols,
                                      _dev(q, torch.int8, "q"), _dev(scale, torch.float32, "scale"),
                                      _stream(stream)), "mla_w8a8_quant_rows")


def mla_w8a8_gemm_s32(A, W, acc, stream=None):
    M, K = A.shape
    K2, N = W.shape
    if K2 != K or tuple(acc.shape) != (M, N):
        raise ValueError("shape mismatch")
    _check(load().mla_w8a8_gemm_s32(_dev(A, torch.int8, "A"), _dev(W, torch.int8, "W"), M, K, N,
                                    _dev(acc, torch.int32, "acc"), _stream(stream)),
           "mla_w8a8_gemm_s32")


def mla_prolog_w8a8_operands(h, T, q1, s1, c1, s2, stream=None):
    _check(load().mla_prolog_w8a8_operands(h, T, _dev(q1, torch.int8, "q1"),
                                           _dev(s1, torch.float32, "s1"),
                                           _dev(c1, torch.int8, "c1"),
                                           _dev(s2, torch.float32, "s2"), _stream(stream)),
           "mla_prolog_w8a8_operands")


def mla_prolog_w8a8_capture(h, acc_a=None, acc_qb=None, acc_kvb=None):
    def opt(t, name):
        return None if t is None else _dev(t, torch.int32, name)
    _check(load().mla_prolog_w8a8_capture(h, opt(acc_a, "acc_a"), opt(acc_qb, "acc_qb"),
                                          opt(acc_kvb, "acc_kvb")), "mla_prolog_w8a8_capture")


# ------------------------------------------------------------------ convenience wrapper
class MLAProlog:
    """Owns one library handle (and so one device workspace)."""

    def __init__(self, cfg: dict, max_tokens: int, spin_budget_ns: int = 0):
        self.cfg = cfg
        self.max_tokens = max_tokens
        self.h = mla_kv_prolog_create(cfg, max_tokens, spin_budget_ns)

    def close(self):
        if self.h is not None:
            mla_kv_prolog_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_path(self, path: int):
        mla_kv_prolog_set_path(self.h, path)

    @property
    def last_launches(self) -> int:
        return load().mla_kv_prolog_last_launches(self.h)

    @property
    def last_path(self) -> int:
        return load().mla_kv_prolog_last_path(self.h)

    @property
    def last_cluster_launches(self) -> int:
        return load().mla_kv_prolog_last_cluster_launches(self.h)

    @property
    def auto_threshold(self) -> int:
        return load().mla_kv_prolog_auto_threshold(self.h)

    def status(self, stream=None) -> int:
        return mla_kv_prolog_status(self.h, stream)

    def prepare_weights(self, d: dict, stream=None):
        """Packed snapshot of d["W_kva"], d["W_kvb"]; runs passing these tensors use it."""
        mla_kv_prolog_prepare_weights(self.h, self.cfg, d["W_kva"], d["W_kvb"], stream)

    def alloc_outputs(self, b: int, s: int, device="cuda"):
        c = self.cfg
        dt = torch.bfloat16 if c.get("quant") == "w8a8" else _tdt(c)
        H = c["num_heads"]
        out = dict(k_nope=torch.empty(b, H, s, c["nope_dim"], dtype=dt, device=device),
                   value=torch.empty(b, H, s, c["v_dim"], dtype=dt, device=device),
                   k_pe=torch.empty(b, 1, s, c["rope_dim"], dtype=dt, device=device))
        if c.get("quant") == "w8a8":
            out["q_nope"] = torch.empty(b, H, s, c["nope_dim"], dtype=dt, device=device)
            out["q_pe"] = torch.empty(b, H, s, c["rope_dim"], dtype=dt, device=device)
        return out

    def alloc_latent_outputs(self, b: int, s: int, device="cuda"):
        c = self.cfg
        dt = _tdt(c)
        return dict(latent=torch.empty(b * s, c["kv_lora_rank"], dtype=dt, device=device),
                    k_pe=torch.empty(b, 1, s, c["rope_dim"], dtype=dt, device=device))

    def run_latent(self, b, s, d: dict, out: dict, stream=None):
        """Latent-cache variant: out["latent"] [b*s, 512] and out["k_pe"]."""
        mla_kv_prolog_run_latent(self.h, self.cfg, b, s, d["hidden"], d["positions"], d["W_kva"],
                                 d["gamma_kv"], d["cos"], d["sin"], out["latent"], out["k_pe"], stream)
        return out

    def alloc_paged_caches(self, num_blocks: int, page_size: int, device="cuda"):
        c = self.cfg
        dt = _tdt(c)
        H = c["num_heads"]
        return dict(k_cache=torch.empty(num_blocks, H, page_size, c["nope_dim"], dtype=dt, device=device),
                    v_cache=torch.empty(num_blocks, H, page_size, c["v_dim"], dtype=dt, device=device),
                    kpe_cache=torch.empty(num_blocks, 1, page_size, c["rope_dim"], dtype=dt, device=device))

    def run_paged(self, b, s, d: dict, slot_mapping, page_size: int, caches: dict, stream=None):
        """Paged variant: rows scattered into caches (alloc_paged_caches) by slot_mapping."""
        nb = caches["k_cache"].shape[0]
        mla_kv_prolog_run_paged(self.h, self.cfg, b, s, d["hidden"], d["positions"], d["W_kva"],
                                d["gamma_kv"], d["W_kvb"], d["cos"], d["sin"], slot_mapping, page_size,
                                nb, caches["k_cache"], caches["v_cache"], caches["kpe_cache"], stream)
        return caches

    def alloc_c8_outputs(self, b: int, s: int, device="cuda"):
        c = self.cfg
        H, i8 = c["num_heads"], torch.int8
        return dict(k_nope=torch.empty(b, H, s, c["nope_dim"], dtype=i8, device=device),
                    value=torch.empty(b, H, s, c["v_dim"], dtype=i8, device=device),
                    k_pe=torch.empty(b, 1, s, c["rope_dim"], dtype=i8, device=device))

    def run_c8(self, b, s, d: dict, scales: dict, out: dict, stream=None):
        """int8 KV-cache outputs (alloc_c8_outputs) with per-channel scales
        scales["k"] [H*128], scales["v"] [H*128], scales["kpe"] [64]."""
        mla_kv_prolog_run_c8(self.h, self.cfg, b, s, d["hidden"], d["positions"], d["W_kva"],
                             d["gamma_kv"], d["W_kvb"], d["cos"], d["sin"], scales["k"], scales["v"],
                             scales["kpe"], out["k_nope"], out["value"], out["k_pe"], stream)
        return out

    def run(self, b, s, d: dict, out: dict, stream=None):
        """d: device tensors keyed as the input generator names them."""
        if self.cfg.get("quant") == "w8a8":
            mla_prolog_w8a8_run(self.h, b, s, d["hidden"], d["positions"], d["W_qa"], d["s_qa"],
                                d["gamma_q"], d["W_qb"], d["s_qb"], d["W_kva"], d["s_kva"],
                                d["gamma_kv"], d["W_kvb"], d["s_kvb"], d["cos"], d["sin"],
                                out["q_nope"], out["q_pe"], out["k_nope"], out["value"],
                                out["k_pe"], stream)
        else:
            mla_kv_prolog_run(self.h, self.cfg, b, s, d["hidden"], d["positions"], d["W_kva"],
                              d["gamma_kv"], d["W_kvb"], d["cos"], d["sin"], out["k_nope"],
                              out["value"], out["k_pe"], stream)
        return out


def to_device(inp: dict, device="cuda") -> dict:
    """Copy the tensors of an input-generator dict to the device (same bits)."""
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
