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
