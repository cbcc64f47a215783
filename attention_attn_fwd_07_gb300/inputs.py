"""Seeded synthetic inputs and the named workloads.

This module is shared by the CUDA path's callers and by the oracle's callers.
It holds no attention arithmetic: only shapes, seeds and random draws.

Every tensor is drawn i.i.d. N(0, 1) in float32 from a seeded
``torch.Generator`` and rounded to bfloat16 (round-to-nearest-even); those
bfloat16 bits are the common input of both sides.  The long-prefill workload
additionally multiplies K by 4 on exactly ceil(0.01 * Nk) key rows per
(batch, head), chosen by ``randperm`` from the same generator; x4 is exact in
bfloat16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    seed: int
    k_boost_frac: float = 0.0
    splits: tuple = field(default=())
    Hkv: int = 0  # K/V heads (grouped-query attention); 0 = H
    dv: int = 0   # head dim of V (and O); 0 = d

    @property
    def kv_heads(self) -> int:
        return self.Hkv or self.H

    @property
    def v_dim(self) -> int:
        return self.dv or self.d

    @property
    def scale(self) -> float:
        """1/sqrt(d), rounded to float32 as the library receives it."""
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32))


# The five workloads of the fused attention forward (seeds 1000 + index).
TINY = Workload("tiny B1 H1 N128 d64 non-causal", 1, 1, 128, 128, 64, False, 1000)
RAGGED_LENGTHS = (1, 31, 32, 33, 1003)
RAGGED_SPLITS = (1, 3, 16)
PREFILL = Workload("prefill B4 H16 N2048 d64 causal", 4, 16, 2048, 2048, 64, True, 1002)
LONG_PREFILL_CAUSAL = Workload("long prefill B2 H32 N8192 d128 causal, K x4 on 1% rows",
                               2, 32, 8192, 8192, 128, True, 1003, k_boost_frac=0.01)
LONG_PREFILL_NONCAUSAL = Workload("long prefill B2 H32 N8192 d128 non-causal, K x4 on 1% rows",
                                  2, 32, 8192, 8192, 128, False, 1003, k_boost_frac=0.01)
DECODE = Workload("decode B16 H32 Nq1 Nk32768 d128 split-KV", 16, 32, 1, 32768, 128, False,
                  1004, splits=(8, 16, 32, 64))
# Grouped-query decode: 8 K/V heads shared by groups of 4 query heads.
DECODE_GQA = Workload("decode GQA B16 H32 Hkv8 Nq1 Nk32768 d128 split-KV", 16, 32, 1, 32768,
                      128, False, 1005, splits=(8, 16, 32, 64), Hkv=8)
# Eight query heads per K/V head (the tensor-core partial kernel's case).
DECODE_GQA8 = Workload("decode GQA B16 H32 Hkv4 Nq1 Nk32768 d128 split-KV", 16, 32, 1, 32768,
                       128, False, 1006, splits=(4, 8, 16), Hkv=4)


# Head dims beyond 64 and 128 (several head dimensions, GPU Engineering
# section 22.5's lab): long causal prefills with the long prefill's bytes
# per (b, h) scaled by d, and a decode at d = 256.
LONG_PREFILL_D96 = Workload("long prefill B2 H32 N8192 d96 causal", 2, 32, 8192, 8192, 96, True,
                            1008)
LONG_PREFILL_D256 = Workload("long prefill B2 H16 N8192 d256 causal", 2, 16, 8192, 8192, 256,
                             True, 1009)
DECODE_D256 = Workload("decode B8 H16 Nq1 Nk32768 d256 split-KV", 8, 16, 1, 32768, 256, False,
                       1010, splits=(8, 16, 32))


def ragged(n: int, causal: bool) -> Workload:
    """Ragged-length edge case: B=3, H=4, d=64, Nq=Nk=n (seed 1001 + n)."""
    tag = "causal" if causal else "non-causal"
    return Workload(f"ragged B3 H4 N{n} d64 {tag}", 3, 4, n, n, 64, causal, 1001 + n)


def make_qkv(w: Workload, device: str | torch.device = "cpu", Nq: int | None = None,
             Nk: int | None = None):
    """Draw q [B, H, Nq, d] and k, v [B, Hkv, Nk, d] as contiguous bfloat16.

    ``Nq``/``Nk`` override the workload's lengths (smaller parity cases that
    keep the same distribution).
    """
    Nq = w.Nq if Nq is None else Nq
    Nk = w.Nk if Nk is None else Nk
    g = torch.Generator(device=device).manual_seed(w.seed)

    def draw(n, heads, dim=w.d):
        out = torch.empty((w.B, heads, n, dim), dtype=torch.bfloat16, device=device)
        for b in range(w.B):  # per batch keeps the float32 temporary small
            out[b] = torch.randn((heads, n, dim), generator=g, device=device,
                                 dtype=torch.float32).to(torch.bfloat16)
        return out

    q, k, v = draw(Nq, w.H), draw(Nk, w.kv_heads), draw(Nk, w.kv_heads, w.v_dim)
    if w.k_boost_frac > 0.0:
        n_boost = math.ceil(w.k_boost_frac * Nk)
        for b in range(w.B):
            for h in range(w.kv_heads):
                rows = torch.randperm(Nk, generator=g, device=device)[:n_boost]
                k[b, h, rows] = k[b, h, rows] * 4
    return q, k, v


def make_dout(w: Workload, device: str | torch.device = "cpu", Nq: int | None = None):
    """Loss gradient on O for the backward pass: dO [B, H, Nq, dv] bfloat16
    (dv = the value head dim), standard normal entries from its own seed (the
    workload's seed + 104729)."""
    Nq = w.Nq if Nq is None else Nq
    g = torch.Generator(device=device).manual_seed(w.seed + 104729)
    out = torch.empty((w.B, w.H, Nq, w.v_dim), dtype=torch.bfloat16, device=device)
    for b in range(w.B):
        out[b] = torch.randn((w.H, Nq, w.v_dim), generator=g, device=device,
                             dtype=torch.float32).to(torch.bfloat16)
    return out


def make_qkv_fp8(w: Workload, device: str | torch.device = "cpu", Nq: int | None = None,
                 Nk: int | None = None):
    """FP8 Q K^T inputs: q, k as e4m3 codes (uint8 tensors) with per-tensor
    descales, v as bfloat16.  The float32 draws of ``make_qkv``'s recipe are
    divided by amax / 448 (e4m3's largest finite value) and rounded to e4m3
    by torch's converter; returns (q8, k8, v, q_descale, k_descale)."""
    Nq = w.Nq if Nq is None else Nq
    Nk = w.Nk if Nk is None else Nk
    g = torch.Generator(device=device).manual_seed(w.seed + 7919)

    def draw(n, heads, width=w.d):
        return torch.randn((w.B, heads, n, width), generator=g, device=device, dtype=torch.float32)

    def quantise(x):
        descale = float(x.abs().max()) / 448.0
        codes = (x / descale).to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
        return codes, descale

    q8, qd = quantise(draw(Nq, w.H))
    k32 = draw(Nk, w.kv_heads)
    if w.k_boost_frac > 0.0:
        n_boost = math.ceil(w.k_boost_frac * Nk)
        for b in range(w.B):
            for h in range(w.kv_heads):
                rows = torch.randperm(Nk, generator=g, device=device)[:n_boost]
                k32[b, h, rows] *= 4
    k8, kd = quantise(k32)
    v = draw(Nk, w.kv_heads, w.v_dim).to(torch.bfloat16)
    return q8, k8, v, qd, kd
