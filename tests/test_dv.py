"""GPU parity for a value head dim different from the key head dim (dv != d,
which the online-softmax derivation allows: V only enters through P V).
Prefill and split-KV paths, d and dv in {64, 128} (the backward's cases
are in test_bwd.py)."""
import pytest
import torch

import oracle
from attention_attn_fwd_07_gb300 import binding, build
from attention_attn_fwd_07_gb300 import inputs as W
from tests.parity_util import compare, check_guards, guarded

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    build.build()
    binding.load_library()
    yield
    assert binding.attn_get_device_status() == 0


def run(q, k, v, causal, scale, query_offset=0):
    B, H, Nq, _ = q.shape
    dv = v.shape[3]
    o, obuf, opad = guarded((B, H, Nq, dv), torch.bfloat16, DEV)
    lse, lbuf, lpad = guarded((B, H, Nq), torch.float32, DEV)
    flags = binding.ATTN_FLAG_ALLOW_NEG_OFFSET if query_offset < 0 else 0
    binding.attn_fwd_ex(q, k, v, causal, scale, query_offset=query_offset, flags=flags, o=o,
                        lse=lse)
    torch.cuda.synchronize()
    check_guards(obuf, opad, "O")
    check_guards(lbuf, lpad, "LSE")
    return o, lse


@pytest.mark.parametrize("d,dv", [(64, 128), (128, 64)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", [1, 129, 333, 1003])
def test_dv_prefill(d, dv, causal, n):
    w = W.Workload("dv", 2, 3, n, n, d, causal, 3000 + n + d, dv=dv)
    q, k, v = W.make_qkv(w)
    assert v.shape[3] == dv
    o, lse = run(*(t.to(DEV) for t in (q, k, v)), causal, w.scale)
    compare(o, lse, *oracle.attention(q, k, v, causal=causal, scale=w.scale),
            f"d={d} dv={dv} N={n} causal={causal}")


@pytest.mark.parametrize("d,dv", [(64, 128), (128, 64)])
def test_dv_gqa_and_offsets(d, dv):
    w = W.Workload("dv gqa", 1, 8, 300, 700, d, True, 3100 + d, Hkv=2, dv=dv)
    q, k, v = W.make_qkv(w)
    for off in (-120, 0, 400):
        o, lse = run(*(t.to(DEV) for t in (q, k, v)), True, w.scale, query_offset=off)
        compare(o, lse, *oracle.attention(q, k, v, causal=True, scale=w.scale, query_offset=off),
                f"d={d} dv={dv} GQA offset={off}")


def test_dv_long_prefill_sampled():
    """Long causal prefill shape with dv = 64 (d = 128): sampled rows."""
    w = W.Workload("dv long", 1, 8, 8192, 8192, 128, True, 3200, dv=64)
    q, k, v = W.make_qkv(w, device=DEV)
    o, lse = run(q, k, v, True, w.scale)
    rows = torch.randint(0, w.H * w.Nq, (96,), generator=torch.Generator().manual_seed(5)).tolist()
    ref_o, ref_l = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True, scale=w.scale,
                                    rows=rows)
    idx = torch.tensor(rows)
    compare(o.reshape(-1, 64)[idx], lse.reshape(-1)[idx], ref_o, ref_l, "dv long sampled")


def run_splitkv(q, k, v, causal, scale, splits, query_offset=0):
    B, H, Nq, _ = q.shape
    dv = v.shape[3]
    o, obuf, opad = guarded((B, H, Nq, dv), torch.bfloat16, DEV)
    lse, lbuf, lpad = guarded((B, H, Nq), torch.float32, DEV)
    flags = binding.ATTN_FLAG_ALLOW_NEG_OFFSET if query_offset < 0 else 0
    binding.attn_fwd_splitkv_ex(q, k, v, causal, scale, splits, query_offset=query_offset,
                                flags=flags, o=o, lse=lse)
    torch.cuda.synchronize()
    check_guards(obuf, opad, "O")
    check_guards(lbuf, lpad, "LSE")
    return o, lse


@pytest.mark.parametrize("d,dv", [(64, 128), (128, 64)])
@pytest.mark.parametrize("nk", [1, 700, 4099])
@pytest.mark.parametrize("splits", [1, 3, 16])
def test_dv_splitkv_decode(d, dv, nk, splits):
    """One query row per head against nk keys (decode), plain and causal at
    the last position."""
    w = W.Workload("dv decode", 2, 4, 1, nk, d, False, 3400 + nk + d + splits, dv=dv)
    q, k, v = W.make_qkv(w)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    o, lse = run_splitkv(qd, kd, vd, False, w.scale, splits)
    compare(o, lse, *oracle.attention(q, k, v, causal=False, scale=w.scale),
            f"split-KV d={d} dv={dv} Nk={nk} S={splits}")
    o, lse = run_splitkv(qd, kd, vd, True, w.scale, splits, query_offset=nk - 1)
    compare(o, lse, *oracle.attention(q, k, v, causal=True, scale=w.scale, query_offset=nk - 1),
            f"split-KV causal d={d} dv={dv} Nk={nk} S={splits}")


@pytest.mark.parametrize("d,dv", [(64, 128), (128, 64)])
def test_dv_splitkv_gqa_rows_and_offsets(d, dv):
    """Grouped K/V heads and several query positions (chunked decode), with
    offsets that leave whole splits, and (negative offset) whole rows,
    without an admissible key."""
    w = W.Workload("dv split gqa", 2, 8, 5, 1000, d, True, 3500 + d, Hkv=2, dv=dv)
    q, k, v = W.make_qkv(w)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    for off in (-3, 0, 400, 995):
        o, lse = run_splitkv(qd, kd, vd, True, w.scale, 6, query_offset=off)
        compare(o, lse, *oracle.attention(q, k, v, causal=True, scale=w.scale, query_offset=off),
                f"split-KV d={d} dv={dv} GQA offset={off}")
