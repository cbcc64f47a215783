"""The seeded input recipe (no GPU): every parity case and bench line draws
its inputs here, so its stated properties are checked directly."""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

from attention_attn_fwd_07_gb300 import inputs as W
from oracle.fp8 import decode_e4m3


def small(w: W.Workload, **kw) -> W.Workload:
    """The same recipe at a size the CPU draws in milliseconds."""
    return dataclasses.replace(w, **kw)


def test_draws_are_seeded_bf16_and_shaped():
    w = small(W.DECODE_GQA, B=2, Nk=300)
    q, k, v = W.make_qkv(w)
    assert q.dtype == k.dtype == v.dtype == torch.bfloat16
    assert q.shape == (2, 32, 1, 128) and k.shape == (2, 8, 300, 128) and v.shape == k.shape
    assert all(t.is_contiguous() for t in (q, k, v))
    q2, k2, v2 = W.make_qkv(w)
    for a, b in ((q, q2), (k, k2), (v, v2)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    q3, _, _ = W.make_qkv(small(w, seed=w.seed + 1))
    assert not torch.equal(q.view(torch.int16), q3.view(torch.int16))


def test_value_dim_and_length_overrides():
    w = W.Workload("dv", 1, 4, 50, 70, 128, False, 7, Hkv=2, dv=64)
    q, k, v = W.make_qkv(w)
    assert q.shape == (1, 4, 50, 128) and k.shape == (1, 2, 70, 128)
    assert v.shape == (1, 2, 70, 64)
    q, k, v = W.make_qkv(w, Nq=5, Nk=9)
    assert q.shape[2] == 5 and k.shape[2] == 9 and v.shape[2] == 9
    assert W.make_dout(w).shape == (1, 4, 50, 64)


def test_standard_normal():
    q, k, v = W.make_qkv(small(W.PREFILL, B=1, H=2, Nq=512, Nk=512))
    x = torch.cat([t.float().flatten() for t in (q, k, v)]).numpy().astype(np.float64)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1.0) < 0.02


def test_k_boost_scales_exactly_one_percent_of_rows_by_four():
    base = small(W.LONG_PREFILL_CAUSAL, B=2, H=3, Nq=16, Nk=1000)
    plain = small(base, k_boost_frac=0.0)
    q, k, v = W.make_qkv(base)
    q0, k0, v0 = W.make_qkv(plain)
    # Q and V, and K away from the boosted rows, are the unboosted draws.
    assert torch.equal(q.view(torch.int16), q0.view(torch.int16))
    assert torch.equal(v.view(torch.int16), v0.view(torch.int16))
    n_boost = math.ceil(0.01 * 1000)
    for b in range(2):
        for h in range(3):
            same = (k[b, h] == k0[b, h]).all(dim=1)
            four = (k[b, h].float() == 4 * k0[b, h].float()).all(dim=1)
            assert int((~same).sum()) == n_boost, (b, h)
            assert bool(four[~same].all())  # x4 is exact in bf16


def test_fp8_codes_and_descales():
    w = small(W.LONG_PREFILL_CAUSAL, B=1, H=2, Nq=64, Nk=200)
    q8, k8, v, qd, kd = W.make_qkv_fp8(w)
    assert q8.dtype == k8.dtype == torch.uint8 and v.dtype == torch.bfloat16
    qv, kv = decode_e4m3(q8.numpy()), decode_e4m3(k8.numpy())
    assert np.isfinite(qv).all() and np.isfinite(kv).all()
    # Each tensor's largest magnitude maps to e4m3's largest finite value.
    assert np.abs(qv).max() == 448.0 and np.abs(kv).max() == 448.0
    assert qd > 0.0 and kd > 0.0


def test_scale_is_the_float32_rounding_of_one_over_sqrt_d():
    for d in (64, 128):
        w = W.Workload("s", 1, 1, 1, 1, d, False, 0)
        assert w.scale == float(np.float32(1.0 / math.sqrt(d)))
