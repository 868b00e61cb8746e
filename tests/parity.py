"""Comparison helpers shared by the GPU parity tests.

Tolerance (per output tensor), for fp16/bf16 outputs: max |g - o_r| <= 2e-2
and sum|g - o_r| / sum|o_r| <= 5e-3, where o_r is the fp64 oracle rounded
to the output dtype (nearest even).  Rounding the oracle first keeps the
bound meaningful for large-magnitude entries, where half an ulp of bf16
already exceeds 2e-2.
"""
import numpy as np
import torch

MAX_ABS = 2e-2
MEAN_REL = 5e-3


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
    assert mx <= max_abs, f"{name}: max |err| {mx:.3e} > {max_abs}"
    assert rel <= mean_rel, f"{name}: mean rel err {rel:.3e} > {mean_rel}"
    return mx, rel, raw
