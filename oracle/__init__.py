"""CPU oracle of the MLA KV prolog (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
binding) never imports it, links it or falls back to it.

The arithmetic lives in ``oracle.c`` (plain C, fp64); this module builds it
with gcc and wraps it with ctypes.  Inputs are passed as the same bits the
GPU receives: 16-bit floats as ``uint16`` arrays (fp16 or bf16 encodings),
int8 weights, fp32 scales and fp32 cos/sin tables.

Sources: "DeepSeek-V2-Lite-Chat MLA KV Prolog 迁移指南" (the seven prolog
steps, §背景; the shapes, §精度验证) and "DeepSeek-R1或Kimi-K2模型在NPU实现高性能
推理" (the W8A8 weight mode, §权重转换).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (OpenMP when available).
    With MLA_ORACLE_SO set, that prebuilt library is used instead (the
    mutation tests load deliberately broken copies this way)."""
    if os.environ.get("MLA_ORACLE_SO"):
        return os.environ["MLA_ORACLE_SO"]
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    os.makedirs(_BUILD, exist_ok=True)
    base = ["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-shared", "-fPIC",
            src, "-lm"]
    tmp = _SO + ".tmp%d" % os.getpid()
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-o", tmp], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-o", tmp], check=True, capture_output=True)
    os.replace(tmp, _SO)
    return _SO


class _Dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int64), ("rank", ctypes.c_int64), ("rope", ctypes.c_int64),
                ("heads", ctypes.c_int64), ("nope", ctypes.c_int64), ("vdim", ctypes.c_int64),
                ("max_pos", ctypes.c_int64), ("eps", ctypes.c_double), ("dtype", ctypes.c_int)]


class _W8Dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int64), ("q_rank", ctypes.c_int64),
                ("kv_rank", ctypes.c_int64), ("rope", ctypes.c_int64),
                ("heads", ctypes.c_int64), ("nope", ctypes.c_int64), ("vdim", ctypes.c_int64),
                ("max_pos", ctypes.c_int64), ("eps", ctypes.c_double)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            L.oracle_f16_to_double.restype = ctypes.c_double
            L.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_double.restype = ctypes.c_double
            L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_double_to_f16.restype = ctypes.c_uint16
            L.oracle_double_to_f16.argtypes = [ctypes.c_double]
            L.oracle_double_to_bf16.restype = ctypes.c_uint16
            L.oracle_double_to_bf16.argtypes = [ctypes.c_double]
            L.oracle_promote16.restype = None
            L.oracle_promote16.argtypes = [P, ctypes.c_int64, ctypes.c_int, P]
            L.oracle_vec_matmul.restype = None
            L.oracle_vec_matmul.argtypes = [P, P, ctypes.c_int64, ctypes.c_int64, P]
            L.oracle_rmsnorm.restype = None
            L.oracle_rmsnorm.argtypes = [P, ctypes.c_int64, P, ctypes.c_double, P]
            L.oracle_rope.restype = None
            L.oracle_rope.argtypes = [P, ctypes.c_int, P, P, P]
            L.oracle_kv_prolog.restype = ctypes.c_int
            L.oracle_kv_prolog.argtypes = [ctypes.POINTER(_Dims), ctypes.c_int64, ctypes.c_int64,
                                           P, P, P, P, P, P, P, P, ctypes.c_int64, ctypes.c_int,
                                           P, P, P]
            L.oracle_kv_latent.restype = ctypes.c_int
            L.oracle_kv_latent.argtypes = [ctypes.POINTER(_Dims), ctypes.c_int64, ctypes.c_int64,
                                           P, P, P, P, P, P, P, ctypes.c_int64, ctypes.c_int, P, P]
            L.oracle_quant_row_f32.restype = None
            L.oracle_quant_row_f32.argtypes = [P, ctypes.c_int64, P, P]
            L.oracle_int_gemm.restype = None
            L.oracle_int_gemm.argtypes = [P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, P]
            L.oracle_w8a8.restype = ctypes.c_int
            L.oracle_w8a8.argtypes = [ctypes.POINTER(_W8Dims), ctypes.c_int64, ctypes.c_int64,
                                      P, P, P, P, P, P, P, P, P, P, P, P, P, P, P,
                                      ctypes.c_int64, ctypes.c_int, P, P, P, P, P]
            L.oracle_w8a8_token_operands.restype = ctypes.c_int
            L.oracle_w8a8_token_operands.argtypes = [ctypes.POINTER(_W8Dims), ctypes.c_int64,
                                                     P, P, P, P, P, P, P, P, P, P, P, P, P, P]
            L.oracle_round_array.restype = None
            L.oracle_round_array.argtypes = [P, ctypes.c_int64, ctypes.c_int, P]
            L.oracle_openmp_max_threads.restype = ctypes.c_int
            L.oracle_openmp_max_threads.argtypes = []
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits16(a) -> np.ndarray:
    """16-bit float tensor/array -> contiguous uint16 view of its bits."""
    if hasattr(a, "view") and hasattr(a, "numpy") and not isinstance(a, np.ndarray):
        import torch
        return a.detach().contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return a


def _np(a, dtype) -> np.ndarray:
    if hasattr(a, "numpy") and not isinstance(a, np.ndarray):
        a = a.detach().contiguous().numpy()
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- scalars
def f16_to_double(bits: int) -> float:
    return lib().oracle_f16_to_double(int(bits))


def bf16_to_double(bits: int) -> float:
    return lib().oracle_bf16_to_double(int(bits))


def double_to_f16(x: float) -> int:
    return lib().oracle_double_to_f16(float(x))


def double_to_bf16(x: float) -> int:
    return lib().oracle_double_to_bf16(float(x))


def promote16(bits, dtype: int) -> np.ndarray:
    """uint16 bits (dtype 0 = fp16, 1 = bf16) -> float64, bit-exact."""
    b = _bits16(bits)
    out = np.empty(b.shape, dtype=np.float64)
    lib().oracle_promote16(_ptr(b), b.size, dtype, _ptr(out))
    return out


def round_to(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round float64 values to fp16 (0) / bf16 (1), nearest-even, and return
    them as float64 (the value of the rounded 16-bit number)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    lib().oracle_round_array(_ptr(x), x.size, dtype, _ptr(out))
    return out


# ---------------------------------------------------------------- steps
def vec_matmul(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    x = _np(x, np.float64)
    W = _np(W, np.float64)
    K, N = W.shape
    y = np.empty(N, dtype=np.float64)
    lib().oracle_vec_matmul(_ptr(x), _ptr(W), K, N, _ptr(y))
    return y


def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    x = _np(x, np.float64)
    g = _np(gamma, np.float64)
    y = np.empty_like(x)
    lib().oracle_rmsnorm(_ptr(x), x.size, _ptr(g), eps, _ptr(y))
    return y


def rope(x: np.ndarray, cos_row: np.ndarray, sin_row: np.ndarray) -> np.ndarray:
    x = _np(x, np.float64)
    c = _np(cos_row, np.float32)
    s = _np(sin_row, np.float32)
    y = np.empty_like(x)
    lib().oracle_rope(_ptr(x), x.size, _ptr(c), _ptr(s), _ptr(y))
    return y


def quant_row_f32(x: np.ndarray):
    x = _np(x, np.float32)
    q = np.empty(x.size, dtype=np.int8)
    s = np.zeros(1, dtype=np.float32)
    lib().oracle_quant_row_f32(_ptr(x), x.size, _ptr(q), _ptr(s))
    return q, float(s[0])


def int_gemm(A: np.ndarray, W: np.ndarray) -> np.ndarray:
    """Brute-force int8 x int8 GEMM with int64 accumulation."""
    A = _np(A, np.int8)
    W = _np(W, np.int8)
    M, K = A.shape
    K2, N = W.shape
    assert K == K2
    acc = np.empty((M, N), dtype=np.int64)
    lib().oracle_int_gemm(_ptr(A), _ptr(W), M, K, N, _ptr(acc))
    return acc


# ---------------------------------------------------------------- whole prolog
def kv_prolog(inp: dict, rows=None, nthreads: int = 0):
    """fp64 KV prolog on the dict made by the input generator.

    Returns (k_nope [b,H,s,128], value [b,H,s,128], k_pe [b,1,s,64]) as
    float64; with ``rows`` only those token rows (t = bi*s + si) are filled,
    the rest are NaN.  Raises if a listed position is out of range."""
    cfg = inp["cfg"]
    b, s = inp["b"], inp["s"]
    T = b * s
    H, dn, dv, dr = cfg["num_heads"], cfg["nope_dim"], cfg["v_dim"], cfg["rope_dim"]
    d = _Dims(cfg["hidden"], cfg["kv_lora_rank"], dr, H, dn, dv, inp["cos"].shape[0],
              cfg["eps"], 0 if cfg["dtype"] == "fp16" else 1)
    hid = _bits16(inp["hidden"])
    pos = _np(inp["positions"], np.int32)
    wa = _bits16(inp["W_kva"])
    g = _bits16(inp["gamma_kv"])
    wb = _bits16(inp["W_kvb"])
    cos = _np(inp["cos"], np.float32)
    sin = _np(inp["sin"], np.float32)
    rows = np.arange(T, dtype=np.int64) if rows is None else _np(rows, np.int64)
    k_nope = np.full((b, H, s, dn), np.nan)
    value = np.full((b, H, s, dv), np.nan)
    k_pe = np.full((b, 1, s, dr), np.nan)
    nt = nthreads if nthreads > 0 else (os.cpu_count() or 1)
    bad = lib().oracle_kv_prolog(ctypes.byref(d), b, s, _ptr(hid), _ptr(pos), _ptr(wa), _ptr(g),
                                 _ptr(wb), _ptr(cos), _ptr(sin), _ptr(rows), rows.size, nt,
                                 _ptr(k_nope), _ptr(value), _ptr(k_pe))
    if bad:
        raise ValueError(f"{bad} token rows have positions outside [0, max_pos)")
    return k_nope, value, k_pe


def kv_latent(inp: dict, rows=None, nthreads: int = 0):
    """fp64 latent-cache variant (steps 1, 2, 3, 6 of the prolog) on the dict
    made by the input generator: (latent [b*s, 512], k_pe [b,1,s,64]) as
    float64; rows not listed in ``rows`` are NaN."""
    cfg = inp["cfg"]
    b, s = inp["b"], inp["s"]
    T = b * s
    r, dr = cfg["kv_lora_rank"], cfg["rope_dim"]
    d = _Dims(cfg["hidden"], r, dr, cfg["num_heads"], cfg["nope_dim"], cfg["v_dim"],
              inp["cos"].shape[0], cfg["eps"], 0 if cfg["dtype"] == "fp16" else 1)
    hid = _bits16(inp["hidden"])
    pos = _np(inp["positions"], np.int32)
    wa = _bits16(inp["W_kva"])
    g = _bits16(inp["gamma_kv"])
    cos = _np(inp["cos"], np.float32)
    sin = _np(inp["sin"], np.float32)
    rows = np.arange(T, dtype=np.int64) if rows is None else _np(rows, np.int64)
    latent = np.full((T, r), np.nan)
    k_pe = np.full((b, 1, s, dr), np.nan)
    nt = nthreads if nthreads > 0 else (os.cpu_count() or 1)
    bad = lib().oracle_kv_latent(ctypes.byref(d), b, s, _ptr(hid), _ptr(pos), _ptr(wa), _ptr(g),
                                 _ptr(cos), _ptr(sin), _ptr(rows), rows.size, nt, _ptr(latent),
                                 _ptr(k_pe))
    if bad:
        raise ValueError(f"{bad} token rows have positions outside [0, max_pos)")
    return latent, k_pe


def quant_c8(x: np.ndarray, scale: np.ndarray, dtype: int) -> np.ndarray:
    """int8 KV-cache codes of prolog outputs x (float64, any shape whose
    last axis is the channel): x is first rounded to the I/O dtype (the value
    the dense output would hold), then, in IEEE float32 operations,
    inv = 1 / scale[c], q = clamp(rint(x * inv), -127, 127).  NaN entries
    (rows not computed) map to 0."""
    xd = round_to(np.nan_to_num(x, nan=0.0), dtype).astype(np.float32)
    inv = (np.float32(1.0) / np.asarray(scale, dtype=np.float32)).astype(np.float32)
    y = (xd * inv).astype(np.float32)
    return np.clip(np.rint(y), -127, 127).astype(np.int8)


def scatter_paged(dense: tuple, b: int, s: int, slots, page_size: int, num_blocks: int):
    """Paged KV-cache layout of the dense prolog outputs (k_nope, value
    [b,H,s,d], k_pe [b,1,s,64]): token row t = bi*s + si goes to slot
    slots[t] = block * page_size + offset, i.e. k_cache[block, h, offset, :]
    (caches [num_blocks, H, page_size, d] and [num_blocks, 1, page_size,
    64]); a negative slot drops the row.  Entries no row writes are NaN."""
    slots = np.asarray(slots, dtype=np.int64)
    outs = []
    for a in dense:
        H, d = a.shape[1], a.shape[3]
        c = np.full((num_blocks, H, page_size, d), np.nan)
        for t in range(b * s):
            if slots[t] < 0:
                continue
            blk, off = divmod(int(slots[t]), page_size)
            bi, si = divmod(t, s)
            c[blk, :, off, :] = a[bi, :, si, :]
        outs.append(c)
    return tuple(outs)


def _w8_dims(inp):
    cfg = inp["cfg"]
    return _W8Dims(cfg["hidden"], cfg["q_lora_rank"], cfg["kv_lora_rank"], cfg["rope_dim"],
                   cfg["num_heads"], cfg["nope_dim"], cfg["v_dim"], inp["cos"].shape[0],
                   cfg["eps"])


def w8a8_prolog(inp: dict, rows=None, nthreads: int = 0):
    """fp64 W8A8 full MLA prolog.  Returns (q_nope, q_pe, k_nope, value,
    k_pe) as float64 in head-major layout; unlisted rows are NaN."""
    cfg = inp["cfg"]
    b, s = inp["b"], inp["s"]
    T = b * s
    H, dn, dv, dr = cfg["num_heads"], cfg["nope_dim"], cfg["v_dim"], cfg["rope_dim"]
    d = _w8_dims(inp)
    a = {k: inp[k] for k in inp}
    hid = _bits16(a["hidden"])
    pos = _np(a["positions"], np.int32)
    arrs = [_np(a["W_qa"], np.int8), _np(a["s_qa"], np.float32), _bits16(a["gamma_q"]),
            _np(a["W_qb"], np.int8), _np(a["s_qb"], np.float32), _np(a["W_kva"], np.int8),
            _np(a["s_kva"], np.float32), _bits16(a["gamma_kv"]), _np(a["W_kvb"], np.int8),
            _np(a["s_kvb"], np.float32), _np(a["cos"], np.float32), _np(a["sin"], np.float32)]
    rows = np.arange(T, dtype=np.int64) if rows is None else _np(rows, np.int64)
    q_nope = np.full((b, H, s, dn), np.nan)
    q_pe = np.full((b, H, s, dr), np.nan)
    k_nope = np.full((b, H, s, dn), np.nan)
    value = np.full((b, H, s, dv), np.nan)
    k_pe = np.full((b, 1, s, dr), np.nan)
    nt = nthreads if nthreads > 0 else (os.cpu_count() or 1)
    bad = lib().oracle_w8a8(ctypes.byref(d), b, s, _ptr(hid), _ptr(pos), *[_ptr(x) for x in arrs],
                            _ptr(rows), rows.size, nt, _ptr(q_nope), _ptr(q_pe), _ptr(k_nope),
                            _ptr(value), _ptr(k_pe))
    if bad:
        raise ValueError(f"{bad} token rows have positions outside [0, max_pos)")
    return q_nope, q_pe, k_nope, value, k_pe


def w8a8_operands(inp: dict, t: int):
    """The int8 operands (and scales) the oracle feeds to q_b_proj and
    kv_b_proj for token row t: (q1 [q_rank], s1, c1 [kv_rank], s2)."""
    cfg = inp["cfg"]
    d = _w8_dims(inp)
    hid = _bits16(inp["hidden"])
    pos = _np(inp["positions"], np.int32)
    q1 = np.empty(cfg["q_lora_rank"], dtype=np.int8)
    c1 = np.empty(cfg["kv_lora_rank"], dtype=np.int8)
    s1 = np.zeros(1, dtype=np.float32)
    s2 = np.zeros(1, dtype=np.float32)
    arrs = [_np(inp["W_qa"], np.int8), _np(inp["s_qa"], np.float32), _bits16(inp["gamma_q"]),
            _np(inp["W_kva"], np.int8), _np(inp["s_kva"], np.float32), _bits16(inp["gamma_kv"]),
            _np(inp["cos"], np.float32), _np(inp["sin"], np.float32)]
    bad = lib().oracle_w8a8_token_operands(ctypes.byref(d), t, _ptr(hid), _ptr(pos),
                                           *[_ptr(x) for x in arrs], _ptr(q1), _ptr(s1),
                                           _ptr(c1), _ptr(s2))
    if bad:
        raise ValueError("position out of range")
    return q1, float(s1[0]), c1, float(s2[0])


def max_threads() -> int:
    return lib().oracle_openmp_max_threads()
