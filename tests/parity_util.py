"""Shared helpers of the parity tests: device round trips and the elementwise error bound.

The bound is the one fixed for this SGEMM study, applied exactly as written:

    |C_gpu_ij - R_ij| <= 1e-4 * (S_ij + |beta * c_ij|)

where R is the oracle's FP64 result and S_ij = sum_k |a_ik b_kj| (also from the oracle).
NaN anywhere fails. A tolerance of 0 (S = 0 and beta * c = 0) demands an exact result.
"""
from __future__ import annotations

import numpy as np
import torch

REL = 1e-4


def bound_check(Cg, R, S, beta, C_in):
    """Return (ok, worst ratio err / tol, number of failing elements, index of worst)."""
    Cg = np.asarray(Cg, dtype=np.float64)
    bc = 0.0 if (beta == 0.0 or C_in is None) else np.abs(
        np.float64(np.float32(beta)) * np.asarray(C_in, dtype=np.float64))
    tol = REL * (S + bc)
    err = np.abs(Cg - R)
    good = err <= tol  # NaN compares False
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(tol > 0, err / np.where(tol > 0, tol, 1.0),
                         np.where(err == 0, 0.0, np.inf))
    ratio = np.where(np.isnan(ratio), np.inf, ratio)
    worst = np.unravel_index(int(np.argmax(ratio)), ratio.shape) if ratio.size else None
    return bool(good.all()), float(ratio.max()) if ratio.size else 0.0, int((~good).sum()), worst


def assert_bound(Cg, R, S, beta, C_in, what=""):
    ok, ratio, nfail, worst = bound_check(Cg, R, S, beta, C_in)
    assert ok, f"{what}: {nfail} elements outside the bound, worst ratio {ratio:.3g} at {worst}"
    return ratio


def to_device_view(x: torch.Tensor, ld: int | None = None, offset: int = 0,
                   fill=float("nan")) -> tuple[torch.Tensor, torch.Tensor]:
    """Copy a CPU (rows x cols) float32 matrix into a device buffer with row stride `ld`
    (default: packed) starting `offset` elements into the buffer. Returns (view, buffer);
    everything in the buffer outside the view holds `fill` (a guard band)."""
    rows, cols = x.shape
    ld = ld or max(cols, 1)
    total = offset + (rows - 1) * ld + cols + 8 if rows and cols else offset + 8
    buf = torch.full((total,), fill, dtype=torch.float32, device="cuda")
    if rows and cols:
        view = buf.as_strided((rows, cols), (ld, 1), offset)
        view.copy_(x.to("cuda"))
    else:
        view = buf.as_strided((rows, cols), (ld, 1), offset)
    return view, buf


def guard_intact(buf: torch.Tensor, view: torch.Tensor, fill=float("nan")) -> bool:
    """True if every element of buf outside the view still holds the fill value."""
    mask = torch.ones(buf.numel(), dtype=torch.bool, device=buf.device)
    rows, cols = view.shape
    if rows and cols:
        idx = (view.storage_offset() + torch.arange(rows, device=buf.device)[:, None] *
               view.stride(0) + torch.arange(cols, device=buf.device)[None, :])
        mask[idx.reshape(-1)] = False
    rest = buf[mask]
    if fill != fill:  # NaN
        return bool(torch.isnan(rest).all())
    return bool((rest == fill).all())
