"""GPU parity for grouped K/V heads (GQA/MQA): K and V carry Hkv heads and
query head h reads K/V head h // (H // Hkv).  Prefill and split-KV paths
against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from attention_attn_fwd_07_gb300 import binding, build
from attention_attn_fwd_07_gb300 import inputs as W
from tests.parity_util import compare
from tests.test_parity import DEV, run_fwd, run_split

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    build.build()
    binding.load_library()
    yield
    assert binding.attn_get_device_status() == 0


def to_dev(*ts):
    return [t.to(DEV) for t in ts]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("hkv", [1, 2, 4])
def test_gqa_prefill(d, causal, hkv):
    w = W.Workload("gqa prefill", 2, 8, 333, 333, d, causal, 300 + hkv, Hkv=hkv)
    q, k, v = W.make_qkv(w)
    assert k.shape[1] == hkv
    o, lse = run_fwd(*to_dev(q, k, v), causal, w.scale)
    compare(o, lse, *oracle.attention(q, k, v, causal=causal, scale=w.scale),
            f"gqa prefill Hkv={hkv} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
def test_gqa_splitkv_offsets(d):
    """Eight rows per K/V head (the tensor-core partial kernel) with offsets
    that leave whole rows (negative) or whole splits without an admissible key."""
    w = W.Workload("gqa split offs", 2, 8, 5, 1000, d, True, 450 + d, Hkv=4)
    q, k, v = W.make_qkv(w)
    for off in (-3, 0, 400, 995):
        ref = oracle.attention(q, k, v, causal=True, scale=w.scale, query_offset=off)
        flags = binding.ATTN_FLAG_ALLOW_NEG_OFFSET if off < 0 else 0
        o, lse = run_split(*to_dev(q, k, v), True, w.scale, 6, query_offset=off, flags=flags)
        compare(o, lse, *ref, f"gqa split d={d} offset={off}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("nq", [1, 3, 37])
@pytest.mark.parametrize("hkv", [1, 2, 8])
def test_gqa_splitkv(d, nq, hkv):
    nk = 1000
    w = W.Workload("gqa split", 2, 8, nq, nk, d, True, 400 + nq + hkv, Hkv=hkv)
    q, k, v = W.make_qkv(w)
    off = nk - nq  # the queries are the last nq positions (decoding-style)
    ref = oracle.attention(q, k, v, causal=True, scale=w.scale, query_offset=off)
    for S in (1, 5, 16):
        o, lse = run_split(*to_dev(q, k, v), True, w.scale, S, query_offset=off)
        compare(o, lse, *ref, f"gqa split Hkv={hkv} Nq={nq} S={S}")
    o, lse = run_fwd(*to_dev(q, k, v), True, w.scale, query_offset=off)
    compare(o, lse, *ref, f"gqa prefill path Hkv={hkv} Nq={nq}")


# Groups of four rows take the CUDA-core partial kernel, groups of eight the
# tensor-core one.
GQA8 = W.DECODE_GQA8


@pytest.mark.parametrize("w,S", [(W.DECODE_GQA, 16), (W.DECODE_GQA, 32), (GQA8, 16)],
                         ids=["g4-S16", "g4-S32", "g8-S16"])
def test_gqa_decode_full_size(w, S):
    q, k, v = W.make_qkv(w, device=DEV)
    o, lse = run_split(q, k, v, w.causal, w.scale, S)
    G = w.H // w.kv_heads
    rng = np.random.default_rng(S)
    for b, hk in [(0, 0), (w.B - 1, w.kv_heads - 1)] + [tuple(x) for x in rng.integers(
            0, [w.B, w.kv_heads], size=(3, 2))]:
        hs = slice(hk * G, (hk + 1) * G)
        qh = q[b:b + 1, hs].cpu()
        kh, vh = k[b:b + 1, hk:hk + 1].cpu(), v[b:b + 1, hk:hk + 1].cpu()
        ref = oracle.attention(qh, kh, vh, causal=False, scale=w.scale)
        compare(o[b:b + 1, hs], lse[b:b + 1, hs], *ref, f"gqa decode b={b} hk={hk} S={S}")


def _sweep_cases(n):
    """Seeded shapes across the split-KV dispatch: rows per K/V head from 1 to
    12 (register-streaming, pipelined and tensor-core partial kernels), both
    head dims, ragged key counts, 1..17 splits, causal with offsets that
    leave rows or splits empty, and value dims different from the key dim."""
    rng = np.random.default_rng(2024)
    cases = []
    for i in range(n):
        d = int(rng.choice([64, 128]))
        G = int(rng.choice([1, 2, 3, 4, 6, 8]))
        Hkv = int(rng.choice([1, 2]))
        Nq = int(rng.choice([1, 1, 2, 3]))
        Nk = int(rng.integers(1, 2500))
        S = int(rng.integers(1, 18))
        causal = bool(rng.integers(0, 2))
        off = int(rng.choice([Nk - Nq, Nk // 2, 0, -2])) if causal else 0
        dv = int(rng.choice([0, 0, 0, 64 if d == 128 else 128]))
        cases.append((i, d, G, Hkv, Nq, Nk, S, causal, off, dv))
    return cases


@pytest.mark.parametrize("i,d,G,Hkv,Nq,Nk,S,causal,off,dv", _sweep_cases(40))
def test_splitkv_dispatch_sweep(i, d, G, Hkv, Nq, Nk, S, causal, off, dv):
    w = W.Workload(f"sweep {i}", 1, G * Hkv, Nq, Nk, d, causal, 5000 + i, Hkv=Hkv, dv=dv)
    q, k, v = W.make_qkv(w)
    ref = oracle.attention(q, k, v, causal=causal, scale=w.scale, query_offset=off)
    flags = binding.ATTN_FLAG_ALLOW_NEG_OFFSET if off < 0 else 0
    qd, kd, vd = to_dev(q, k, v)
    if dv:
        o, lse = binding.attn_fwd_splitkv_ex(qd, kd, vd, causal, w.scale, S, query_offset=off,
                                             flags=flags)
        torch.cuda.synchronize()
    else:
        o, lse = run_split(qd, kd, vd, causal, w.scale, S, query_offset=off, flags=flags)
    compare(o, lse, *ref, f"sweep {i}: d={d} G={G} Hkv={Hkv} Nq={Nq} Nk={Nk} S={S} "
                          f"causal={causal} off={off} dv={dv}")
