"""Comparison helpers shared by the GPU parity tests.

Tolerance (per output tensor), for fp16/bf16 outputs: max |g - o_r| <= 2e-2
and sum|g - o_r| / sum|o_r| <= 5e-3, where o_r is the fp64 oracle rounded
to the output dtype (nearest even).  Rounding the oracle first keeps the
bound meaningful for large-magnitude entries, where half an ulp of bf16
already exceeds 2e-2.

Where the dtype's grid spacing at |o_r| is itself wider than 2e-2 (bf16 at
|x| >= 4, fp16 at |x| >= 32), an element may sit on the neighbouring grid
point instead: its exact value lies so close to a rounding midpoint that
the fp32 arithmetic of any kernel can round it the other way.  There the
bound is one grid step, and such elements must stay rare (at most
FLIP_FRAC of the compared elements); the mean relative error bound holds
for every element as before.
"""
import numpy as np
import torch

MAX_ABS = 2e-2
MEAN_REL = 5e-3
FLIP_FRAC = 1e-3


def grid_step(x: np.ndarray, code: int) -> np.ndarray:
    """Spacing of the fp16 (code 0) / bf16 (code 1) grid at |x| (normal
    range): 2^(floor(log2|x|) - mantissa bits)."""
    mant = 10 if code == 0 else 7
    ax = np.maximum(np.abs(x), 1e-30)
    return np.exp2(np.floor(np.log2(ax)) - mant)


def dtype_code(t: torch.Tensor) -> int:
    return 0 if t.dtype == torch.float16 else 1


def compare(name, gpu: torch.Tensor, ref: np.ndarray, oracle_mod, max_abs=MAX_ABS,
            mean_rel=MEAN_REL):
    """Compare a device output with the fp64 oracle on the entries where the
    oracle is defined (not NaN).  Returns (max_abs_err, mean_rel_err,
    max_abs_err_vs_unrounded)."""
    g = gpu.detach().float().cpu().double().numpy()
    assert g.shape == ref.shape, (name, g.shape, ref.shape)
    m = ~np.isnan(ref)
    assert m.any(), name
    o_r = oracle_mod.round_to(ref, dtype_code(gpu))
    assert np.all(np.isfinite(g[m])), f"{name}: non-finite GPU output"
    d = np.abs(g[m] - o_r[m])
    mx = float(d.max())
    rel = float(d.sum() / max(np.abs(o_r[m]).sum(), 1e-300))
    raw = float(np.abs(g[m] - ref[m]).max())
    over = d > max_abs
    if over.any():
        step = grid_step(o_r[m][over], dtype_code(gpu))
        assert np.all(step > max_abs) and np.all(d[over] <= step), \
            f"{name}: max |err| {mx:.3e} > {max_abs} (not a one-step flip where the grid is wider)"
        assert over.sum() <= FLIP_FRAC * d.size, f"{name}: {int(over.sum())} one-step flips of {d.size}"
    assert rel <= mean_rel, f"{name}: mean rel err {rel:.3e} > {mean_rel}"
    return mx, rel, raw
