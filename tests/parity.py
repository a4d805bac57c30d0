"""Element-wise comparison of a GPU result with the oracle.

Error metric (normalised by the per-element sum of |a||b|):
  fp32 output     : |D - D_ref| <= tol * S
  16-bit output   : |D - RNE(D_ref)| <= ulp_out(max(|D|, |RNE(D_ref)|)) + tol * S
                    (the GPU rounds its fp32 sum once, the oracle rounds the exact
                    sum once: the two roundings can differ by one output ulp)
  S == 0          : D must be exactly 0
  integer inputs  : D == RNE(D_ref) bit for bit (every partial sum is exact in fp32)
Tolerances: 2e-3 for 16-bit inputs, 2e-2 for block-scaled fp8, 4e-3 for tf32:
the tensor core keeps 10 of fp32's 23 mantissa bits of each input, so each
product may be off by up to about 2 * 2^-10 relative (2^-9 = 1.95e-3 of S),
plus fp32 accumulation; 4e-3 leaves room for both.
"""
from __future__ import annotations

import numpy as np

import oracle

TOL_16BIT = 2e-3
TOL_FP8 = 2e-2
TOL_TF32 = 4e-3
MANTISSA = {"f32": 23, "bf16": 7, "f16": 10}
MIN_NORMAL_EXP = {"f32": -126, "bf16": -126, "f16": -14}


def ulp(dtype: str, x: np.ndarray) -> np.ndarray:
    """Spacing of the output format at |x| (subnormal spacing below the normal range)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, MIN_NORMAL_EXP[dtype])
    return np.exp2(e - MANTISSA[dtype])


def compare(d_gpu: np.ndarray, dref: np.ndarray, sabs: np.ndarray, out_dtype: str, tol: float,
            exact: bool = False) -> dict:
    d_gpu = np.asarray(d_gpu, dtype=np.float64)
    expect = oracle.round_to(out_dtype, dref)
    if exact:
        bad = d_gpu != expect
        return {"ok": not bad.any(), "mismatches": int(bad.sum()),
                "max_err": float(np.max(np.abs(d_gpu - expect), initial=0)),
                "first_bad": [tuple(int(i) for i in ix) for ix in np.argwhere(bad)[:8]]}
    zero = sabs == 0
    if out_dtype == "f32":
        err = np.abs(d_gpu - dref)
        allowed = tol * sabs
    else:
        err = np.abs(d_gpu - expect)
        allowed = ulp(out_dtype, np.maximum(np.abs(d_gpu), np.abs(expect))) + tol * sabs
    ok_nonzero = (err <= allowed) | zero
    ok_zero = ~zero | (d_gpu == 0)
    ok = ok_nonzero & ok_zero & np.isfinite(d_gpu)
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(zero, 0.0, np.abs(d_gpu - dref) / np.where(zero, 1.0, sabs))
    return {"ok": bool(ok.all()), "mismatches": int((~ok).sum()), "max_rel_err": float(np.max(rel, initial=0.0)),
            "first_bad": [tuple(int(i) for i in ix) for ix in np.argwhere(~ok)[:8]]}


def dump_on_failure(name: str, **arrays) -> None:
    """Save arrays of a failed comparison into the folder named by $DGB_DUMP_DIR
    (when set and existing), for offline inspection."""
    import os
    out = os.environ.get("DGB_DUMP_DIR", "")
    if out and os.path.isdir(out):
        np.savez_compressed(os.path.join(out, "parity_fail_%s.npz" % name), **arrays)
