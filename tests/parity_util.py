"""Comparison of the CUDA path's outputs with the fp64 oracle.

Tolerances (stated by the build's target and restated here):
  * O (bfloat16 output): |O_gpu - O_ref| - half_ulp_bf16(O_ref) <= 1e-2.  The
    half-ulp allowance is the rounding of the exact value to bf16 itself
    (0.0078 for |O| in [2, 4), 0.0156 in [4, 8)); where |O_ref| < 2 the raw
    error must also be <= 1e-2.
  * LSE (float32): |LSE_gpu - LSE_ref| <= 1e-3.
  * Rows with no admissible key: O exactly +0.0 (bits 0x0000), LSE exactly
    -inf.  No NaN anywhere.
"""
from __future__ import annotations

import numpy as np
import torch

O_TOL = 1e-2
LSE_TOL = 1e-3


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax >= 2.0 ** -126, 2.0 ** (e - 8), 2.0 ** -134)


def compare(o_gpu: torch.Tensor, lse_gpu: torch.Tensor, o_ref: np.ndarray, lse_ref: np.ndarray,
            what: str = "") -> dict:
    """Compare one set of rows; shapes [..., d] / [...] must match."""
    o_bits = o_gpu.detach().cpu().contiguous()
    o = o_bits.to(torch.float64).numpy()
    lse = lse_gpu.detach().cpu().to(torch.float64).numpy()
    assert o.shape == o_ref.shape, f"{what}: O shape {o.shape} vs {o_ref.shape}"
    assert lse.shape == lse_ref.shape, f"{what}: LSE shape {lse.shape} vs {lse_ref.shape}"
    assert not np.isnan(o).any(), f"{what}: NaN in O"
    assert not np.isnan(lse).any(), f"{what}: NaN in LSE"

    masked = np.isneginf(lse_ref)
    if masked.any():
        raw = o_bits.view(torch.int16).numpy()[masked]
        assert (raw == 0).all(), f"{what}: fully masked rows must be +0.0 bits"
        assert np.isneginf(lse[masked]).all(), f"{what}: fully masked rows must have LSE -inf"
    live = ~masked
    assert np.isfinite(lse[live]).all(), f"{what}: non-finite LSE on a live row"
    err_o = np.abs(o[live] - o_ref[live])
    excess = err_o - half_ulp_bf16(o_ref[live])
    err_l = np.abs(lse[live] - lse_ref[live])
    small = np.abs(o_ref[live]) < 2.0
    stats = {
        "o_max_abs": float(err_o.max()) if err_o.size else 0.0,
        "o_max_excess": float(excess.max()) if excess.size else 0.0,
        "lse_max_abs": float(err_l.max()) if err_l.size else 0.0,
        "rows": int(lse_ref.size),
        "masked_rows": int(masked.sum()),
    }
    assert stats["o_max_excess"] <= O_TOL, f"{what}: O excess {stats}"
    if small.any():
        assert err_o[small].max() <= O_TOL, f"{what}: O raw error {err_o[small].max()}"
    assert stats["lse_max_abs"] <= LSE_TOL, f"{what}: LSE {stats}"
    return stats


def guarded(shape, dtype, device, pad: int = 256):
    """A tensor of `shape` inside a buffer with `pad` sentinel elements on each
    side; returns (view, buffer, sentinel) for checking writes stay in bounds."""
    n = int(np.prod(shape))
    buf = torch.empty(n + 2 * pad, dtype=dtype, device=device)
    if dtype == torch.bfloat16:
        buf.view(torch.int16).fill_(0x7FA5)   # a NaN pattern the kernels never write
    else:
        buf.view(torch.int32).fill_(0x7FC0DEAD)
    view = buf[pad:pad + n].view(shape)
    return view, buf, pad


def check_guards(buf: torch.Tensor, pad: int, what: str = "") -> None:
    raw = buf.view(torch.int16 if buf.dtype == torch.bfloat16 else torch.int32).cpu()
    sentinel = 0x7FA5 if buf.dtype == torch.bfloat16 else 0x7FC0DEAD
    assert (raw[:pad] == sentinel).all(), f"{what}: write before the output"
    assert (raw[-pad:] == sentinel).all(), f"{what}: write after the output"
