"""Shared helpers of the GPU parity tests: run the CUDA path and the oracle on the
same seeded bytes and compare element by element."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as W

# Tolerances (per element).  bf16 outputs: |y - ref| <= 1e-3 + 8e-3 |ref| (one bf16
# ulp is at most 2^-7 |ref|).  fp32 FMA: 1e-5 + 1e-5 |ref|.  tf32: |y - ref| <=
# 2e-3 * max |ref| over the token's row of that projection (tf32 operand error
# scales with the terms, not with the result), plus a normwise 2e-3.
BF16_ATOL, BF16_RTOL = 1e-3, 8e-3
FP32_ATOL, FP32_RTOL = 1e-5, 1e-5
TF32_ROWMAX_REL = 2e-3


def oracle_outputs(x: torch.Tensor, w_cat: torch.Tensor, splits, threads: int = 8):
    dt = oracle.BF16 if x.dtype == torch.bfloat16 else oracle.FP32
    outs = oracle.fused(W.to_numpy_bits(x), W.to_numpy_bits(w_cat), splits, dt, threads=threads)
    return [W.from_numpy_bits(o).to(torch.float64).numpy() for o in outs]


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


# Largest element error as a fraction of the allowed band, per checked case and mode
# (printed at the end of the test session by conftest.py), so that a regression that
# still fits inside a band is visible.
MARGINS = []


def check_close(gpu_outs, ref_outs, mode: str, what: str = ""):
    """mode: 'bf16' | 'fp32' | 'tf32'.  Returns the largest error / band over all outputs."""
    worst = 0.0
    for i, (g, r) in enumerate(zip(gpu_outs, ref_outs)):
        g = as_f64(g)
        assert g.shape == r.shape, (what, i, g.shape, r.shape)
        assert np.all(np.isfinite(g)), f"{what} split {i}: non-finite output"
        if mode == "bf16":
            bound = BF16_ATOL + BF16_RTOL * np.abs(r)
        elif mode == "fp32":
            bound = FP32_ATOL + FP32_RTOL * np.abs(r)
        else:
            rowmax = np.max(np.abs(r), axis=1, keepdims=True)
            bound = TF32_ROWMAX_REL * rowmax + 1e-30
            nrm = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
            assert nrm <= TF32_ROWMAX_REL, f"{what} split {i}: normwise {nrm:.3e}"
        err = np.abs(g - r)
        if err.size:
            worst = max(worst, float(np.max(err / bound)))
        bad = err > bound
        if bad.any():
            idx = np.argwhere(bad)[:5]
            detail = ", ".join(f"[{a},{b}] gpu={g[a, b]!r} ref={r[a, b]!r}" for a, b in idx)
            raise AssertionError(f"{what} split {i}: {int(bad.sum())}/{bad.size} outside tolerance; {detail}")
    MARGINS.append((mode, what, worst))
    return worst


def mode_of(dtype: str, tf32: bool) -> str:
    if dtype == "bf16":
        return "bf16"
    return "tf32" if tf32 else "fp32"
