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

import concurrent.futures as cf

import numpy as np
import torch

O_TOL = 1e-2
LSE_TOL = 1e-3
# Relative rounding of one bf16 staging of P: bf16 carries 8 significant
# bits, so round-to-nearest is within 2^-8 of the value; with 1/16 of slack
# for the fp32 accumulations and the exp2 approximation on the same path.
P_ROUND = 2.0 ** -8 * 1.0625


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax >= 2.0 ** -126, 2.0 ** (e - 8), 2.0 ** -134)


def compare(o_gpu: torch.Tensor, lse_gpu: torch.Tensor, o_ref: np.ndarray, lse_ref: np.ndarray,
            what: str = "", absv_ref: np.ndarray | None = None) -> dict:
    """Compare one set of rows; shapes [..., d] / [...] must match.

    ``absv_ref`` (optional, same shape as ``o_ref``) is the oracle's
    attention output with |V| in place of V, i.e. sum_j w_j |v_jc| for the
    exact weights w.  With it, every element must also meet the bound of the
    kernel's own arithmetic: the kernel forms O from P rounded once to bf16
    (each weight off by at most 2^-8 of itself; the row's largest weight is
    rounded too, because its exponent reference may trail the row maximum)
    and rounds the result to bf16, so
    |O_gpu - O_ref| <= half_ulp + 2^-8 sum_j w_j |v_jc| (+ slack),
    half_ulp taken at the larger of |O_ref| and |O_gpu|.  That bound replaces the raw 1e-2 rule on |O_ref| < 2, which a
    row whose few dominant weights sit on large |v| with cancelling signs
    can exceed by the weight rounding alone."""
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
    if absv_ref is not None:
        # The final rounding to bf16 moves the kernel's fp32 value by at most
        # half an ulp at the rounded value's binade (which is the larger one
        # when the value crosses a power of two), hence the ulp of the output.
        ulp_term = np.maximum(half_ulp_bf16(o_ref[live]), half_ulp_bf16(o[live]))
        over = err_o - (ulp_term + P_ROUND * absv_ref[live] + 1e-5)
        stats["o_max_over_bound"] = float(over.max()) if over.size else 0.0
        stats["o_raw_max_small"] = float(err_o[small].max()) if small.any() else 0.0
        if over.size:
            at = np.unravel_index(int(np.argmax(over)), over.shape)
            stats["worst"] = {"o_ref": float(o_ref[live][at]), "o_gpu": float(o[live][at]),
                              "sum_w_absv": float(absv_ref[live][at])}
        assert stats["o_max_over_bound"] <= 0.0, f"{what}: O beyond the bf16-P bound {stats}"
    elif small.any():
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


# Backward tolerance.  Every gradient element is an fp32 sum of products whose
# one staged factor (P for dV, dS for dK and dQ) was rounded to bf16 (relative
# error <= 2^-8, bf16's unit roundoff), and the result is rounded to bf16 once
# more (<= 2^-8 of itself); the row correction comes from the bf16 O.
# Together that stays below 2 * 2^-8 ~ 7.8e-3 of the largest terms, so with
# u = 1e-2:
#   * normwise  ||G - R||_F <= u * ||R||_F      (each of dQ, dK, dV)
#   * per element |G - R| <= half_ulp_bf16(R) + u * max|R|
#   * exact zeros: rows with no admissible key have dQ == 0 and keys that no
#     row sees have dK == dV == 0 (compared as values: -0.0 counts as zero).
# Plus an absolute floor for the one cancellation in the path, dP - Delta in
# fp32: its rounding is 2^-24 x (|dP| + |Delta|), and for unit-normal inputs
# at d = 128 those stay below ~160, so ~1e-5 (this is what is left where the
# exact dS is 0, e.g. a single visible key, where P = 1 and dP = Delta).
GRAD_TOL = 1e-2
GRAD_ATOL = 1e-5


def compare_grad(g_gpu: torch.Tensor, ref: np.ndarray, what: str = "",
                 zero_rows: np.ndarray | None = None) -> dict:
    g = g_gpu.detach().cpu().to(torch.float64).numpy()
    assert g.shape == ref.shape, f"{what}: shape {g.shape} vs {ref.shape}"
    assert np.isfinite(g).all(), f"{what}: non-finite gradient"
    err = np.abs(g - ref)
    rmax = float(np.abs(ref).max()) if ref.size else 0.0
    fro_ref = float(np.linalg.norm(ref.ravel()))
    fro_err = float(np.linalg.norm(err.ravel()))
    excess = err - half_ulp_bf16(ref) - GRAD_TOL * rmax - GRAD_ATOL
    stats = {"max_abs": float(err.max()) if err.size else 0.0, "ref_max": rmax,
             "rel_fro": fro_err / fro_ref if fro_ref > 0 else fro_err,
             "max_excess": float(excess.max()) if excess.size else 0.0}
    if zero_rows is not None and zero_rows.any():
        assert (g[zero_rows] == 0).all(), f"{what}: rows that must be zero are not"
        assert (ref[zero_rows] == 0).all(), f"{what}: oracle rows that must be zero are not"
    assert stats["max_excess"] <= 0.0, f"{what}: element error {stats}"
    assert fro_err <= GRAD_TOL * fro_ref + GRAD_ATOL * np.sqrt(max(ref.size, 1)), \
        f"{what}: normwise error {stats}"
    return stats


def whole_head_grads(oracle, q, k, v, dout, b, h, scale, chunk=512):
    """fp64 dQ, dK, dV of one (b, h) slice (K/V head = query head) from the
    oracle, computed in query-row chunks in parallel: rows [r0, r0 + chunk)
    with query_offset = r0 are that chunk's own causal problem, its dQ rows
    are final and its dK, dV are that chunk's contributions, which sum over
    the chunks (dK_j and dV_j are sums over query rows)."""
    qs, ds = q[b:b + 1, h:h + 1].cpu(), dout[b:b + 1, h:h + 1].cpu()
    ks, vs = k[b:b + 1, h:h + 1].cpu(), v[b:b + 1, h:h + 1].cpu()
    Nq = qs.shape[2]
    starts = list(range(0, Nq, chunk))

    def one(r0):
        sl = slice(r0, min(Nq, r0 + chunk))
        return oracle.attention_bwd(qs[:, :, sl], ks, vs, ds[:, :, sl], causal=True,
                                    scale=scale, query_offset=r0, threads=1)

    with cf.ThreadPoolExecutor(max_workers=min(len(starts), oracle.default_threads())) as ex:
        parts = list(ex.map(one, starts))
    rq = np.concatenate([p[0] for p in parts], axis=2)
    rk = sum(p[1] for p in parts)
    rv = sum(p[2] for p in parts)
    return rq, rk, rv
