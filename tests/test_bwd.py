"""GPU parity of the backward pass (dQ, dK, dV) against the fp64 oracle.

The CUDA side runs the product path a user runs: the prefill kernel's O and
LSE, then attn_bwd.  The oracle recomputes everything from q, k, v and dO in
fp64 (its row correction from the definition rowsum(P * dP), not from O).
Cases span several 128-row tiles with ragged tails, causal and not, grouped
K/V heads, value head dims different from the key head dim, decode-style
and negative query offsets (rows with no admissible
key, keys no row sees), and the full-size workloads: one whole (b, h) slice
compared element by element on dQ, dK and dV, dQ on sampled row blocks of
other slices, and dK and dV of every slice through identities that hold at
any size.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_attn_fwd_07_gb300 import binding, build
from attention_attn_fwd_07_gb300 import inputs as W
from tests.parity_util import check_guards, compare_grad, guarded, whole_head_grads

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


def run_bwd(q, k, v, dout, causal, scale, query_offset=0):
    """Forward then backward on the device; gradients in guarded buffers."""
    flags = binding.ATTN_FLAG_ALLOW_NEG_OFFSET if query_offset < 0 else 0
    o, lse = binding.attn_fwd_ex(q, k, v, causal, scale, query_offset=query_offset, flags=flags)
    dq, qbuf, qpad = guarded(tuple(q.shape), torch.bfloat16, DEV)
    dk, kbuf, kpad = guarded(tuple(k.shape), torch.bfloat16, DEV)
    dv, vbuf, vpad = guarded(tuple(v.shape), torch.bfloat16, DEV)
    need = binding.attn_bwd_workspace_bytes(q.shape[0], q.shape[1], q.shape[2])
    ws = torch.empty((need,), dtype=torch.uint8, device=DEV)
    binding.attn_bwd(q, k, v, o, lse, dout, causal, scale, query_offset=query_offset,
                     flags=flags, workspace=ws, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    for buf, pad, name in ((qbuf, qpad, "dQ"), (kbuf, kpad, "dK"), (vbuf, vpad, "dV")):
        check_guards(buf, pad, name)
    return dq, dk, dv


def masks(B, H, Hkv, Nq, Nk, causal, off):
    """Rows with no admissible key, keys that no row sees (per K/V head)."""
    i = np.arange(Nq)
    j = np.arange(Nk)
    if causal:
        dead_rows = (i + off) < 0
        seen = j <= (Nq - 1 + off)
    else:
        dead_rows = np.zeros(Nq, bool)
        seen = np.ones(Nk, bool)
    zq = np.broadcast_to(dead_rows, (B, H, Nq))
    zk = np.broadcast_to(~seen, (B, Hkv, Nk))
    return zq, zk


def check_case(B, H, Hkv, Nq, Nk, causal, off, seed, what, d=128, dv=0):
    w = W.Workload(what, B, H, Nq, Nk, d, causal, seed, Hkv=Hkv, dv=dv)
    q, k, v = W.make_qkv(w)
    dout = W.make_dout(w)
    dq, dk, dv = run_bwd(*(t.to(DEV) for t in (q, k, v, dout)), causal, w.scale, off)
    rq, rk, rv = oracle.attention_bwd(q, k, v, dout, causal=causal, scale=w.scale,
                                      query_offset=off)
    zq, zk = masks(B, H, Hkv, Nq, Nk, causal, off)
    return (compare_grad(dq, rq, f"{what} dQ", zq), compare_grad(dk, rk, f"{what} dK", zk),
            compare_grad(dv, rv, f"{what} dV", zk))


@pytest.mark.parametrize("d", [64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", [1, 100, 128, 129, 333])
def test_bwd_square(n, causal, d):
    check_case(2, 3, 3, n, n, causal, 0, 2000 + n + d, f"bwd N{n} d={d} causal={causal}", d=d)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk", [(37, 1000), (300, 77), (256, 513)])
def test_bwd_rectangular(nq, nk, causal):
    off = nk - nq if causal else 0
    check_case(1, 2, 2, nq, nk, causal, off, 2100 + nq + nk, f"bwd {nq}x{nk} off={off}")


@pytest.mark.parametrize("d", [64, 96, 128])
@pytest.mark.parametrize("hkv", [1, 2, 4])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_gqa(hkv, causal, d):
    check_case(2, 8, hkv, 200, 270, causal, 0, 2200 + hkv + d,
               f"bwd GQA Hkv={hkv} d={d} causal={causal}", d=d)


@pytest.mark.parametrize("d", [64, 96, 128])
@pytest.mark.parametrize("off", [-150, -1, 5, 400])
def test_bwd_offsets(off, d):
    # off < 0: the first -off rows see no key (dQ = 0) and the last keys no
    # row (dK = dV = 0); off >= Nk - Nq: every key visible to every row.
    check_case(1, 2, 2, 300, 300, True, off, 2300 + off + d, f"bwd causal off={off} d={d}", d=d)


@pytest.mark.parametrize("d,dv", [(64, 128), (128, 64)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", [1, 129, 333])
def test_bwd_value_dim(n, causal, d, dv):
    """Value head dim different from the key head dim."""
    check_case(2, 3, 3, n, n, causal, 0, 8100 + n + d, f"bwd d={d} dv={dv} N={n}", d=d, dv=dv)


@pytest.mark.parametrize("d,dv", [(64, 128), (128, 64)])
def test_bwd_value_dim_gqa_offsets(d, dv):
    for off in (-40, 0, 300):
        check_case(1, 4, 2, 200, 500, True, off, 8200 + d, f"bwd d={d} dv={dv} off={off}",
                   d=d, dv=dv)


def check_whole_head(w, q, k, v, dout, dq, dk, dv, b, h):
    rq, rk, rv = whole_head_grads(oracle, q, k, v, dout, b, h, w.scale)
    for name, g, r in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        compare_grad(g[b:b + 1, h:h + 1], r, f"{w.name}: whole head b={b} h={h} {name}")


def test_bwd_rejects_unsupported_head_dims():
    """Head dim 96 runs with value dim 96 only; 256 has no backward."""
    for d, dv in ((96, 64), (64, 96), (256, 256)):
        w = W.Workload(f"d{d} dv{dv}", 1, 1, 64, 64, d, False, 7, dv=dv)
        q, k, v = (t.to(DEV) for t in W.make_qkv(w))
        o = torch.zeros_like(q[..., :1].expand(*q.shape[:3], v.shape[-1])).contiguous()
        lse = torch.zeros((1, 1, 64), dtype=torch.float32, device=DEV)
        with pytest.raises(binding.AttnError) as e:
            binding.attn_bwd(q, k, v, o, lse, torch.zeros_like(o), False, w.scale)
        assert e.value.status == binding.ATTN_ERR_UNSUPPORTED


def test_bwd_d96_long_prefill_whole_head():
    """B2 H32 N8192 d96 causal (the d = 96 long prefill): the last (b, h)
    slice whole, element by element on dQ, dK and dV, and dK, dV of every
    slice through the softmax identities."""
    w = W.LONG_PREFILL_D96
    q, k, v = W.make_qkv(w, device=DEV)
    dout = W.make_dout(w, device=DEV)
    dq, dk, dv = run_bwd(q, k, v, dout, True, w.scale)
    check_whole_head(w, q, k, v, dout, dq, dk, dv, w.B - 1, w.H - 1)
    sum_dk, sum_dv = dk.double().sum(dim=2), dv.double().sum(dim=2)
    sum_do = dout.double().sum(dim=2)
    assert (sum_dk.abs() <= 1e-2 * dk.double().abs().sum(dim=2) + 1e-3).all()
    assert ((sum_dv - sum_do).abs() <= 1e-2 * dv.double().abs().sum(dim=2) + 1e-3).all()


def test_bwd_d64_prefill_sampled():
    """B4 H16 N2048 d64 causal (the d = 64 prefill workload): two whole (b, h)
    slices (the last one among them) element by element, dQ on sampled row
    blocks of others, dK and dV of every slice through the softmax
    identities."""
    w = W.PREFILL
    q, k, v = W.make_qkv(w, device=DEV)
    dout = W.make_dout(w, device=DEV)
    dq, dk, dv = run_bwd(q, k, v, dout, True, w.scale)
    for b, h in ((w.B - 1, w.H - 1), (1, 5)):
        check_whole_head(w, q, k, v, dout, dq, dk, dv, b, h)
    rng = np.random.default_rng(2600)
    for _ in range(3):
        b, h = int(rng.integers(w.B)), int(rng.integers(w.H))
        r0 = int(rng.integers(w.Nq // 128)) * 128
        sl = slice(r0, r0 + 128)
        rq, _, _ = oracle.attention_bwd(q[b:b + 1, h:h + 1, sl].cpu(), k[b:b + 1, h:h + 1].cpu(),
                                        v[b:b + 1, h:h + 1].cpu(), dout[b:b + 1, h:h + 1, sl].cpu(),
                                        causal=True, scale=w.scale, query_offset=r0)
        compare_grad(dq[b:b + 1, h:h + 1, sl], rq, f"d64 dQ b={b} h={h} rows {r0}+128")
    sum_dk, sum_dv = dk.double().sum(dim=2), dv.double().sum(dim=2)
    sum_do = dout.double().sum(dim=2)
    assert (sum_dk.abs() <= 1e-2 * dk.double().abs().sum(dim=2) + 1e-3).all()
    assert ((sum_dv - sum_do).abs() <= 1e-2 * dv.double().abs().sum(dim=2) + 1e-3).all()


def test_bwd_deterministic():
    w = W.Workload("det", 2, 4, 400, 400, 128, True, 2400, Hkv=2)
    q, k, v = (t.to(DEV) for t in W.make_qkv(w))
    dout = W.make_dout(w).to(DEV)
    a = run_bwd(q, k, v, dout, True, w.scale)
    b = run_bwd(q, k, v, dout, True, w.scale)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_bwd_long_prefill_full_size():
    """B2 H32 N8192 d128 causal (1% of keys x4): the last (b, h) slice whole,
    element by element on dQ, dK and dV (a misplaced or swapped key tile
    fails here); dQ on sampled 128-row blocks of other slices (rows i of head
    h need only q_i, dO_i and all of K, V, so the oracle runs on the row block
    with query_offset = its first row); dK and dV of every slice through the
    softmax identities sum_j dS_ij = 0 and sum_j P_ij = 1, which give, per
    K/V head, sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i over the head's
    query rows."""
    w = W.LONG_PREFILL_CAUSAL
    q, k, v = W.make_qkv(w, device=DEV)
    dout = W.make_dout(w, device=DEV)
    dq, dk, dv = run_bwd(q, k, v, dout, True, w.scale)
    check_whole_head(w, q, k, v, dout, dq, dk, dv, w.B - 1, w.H - 1)
    rng = np.random.default_rng(2500)
    for _ in range(3):
        b, h = int(rng.integers(w.B)), int(rng.integers(w.H))
        r0 = int(rng.integers(w.Nq // 128)) * 128
        sl = slice(r0, r0 + 128)
        qs, ds = q[b:b + 1, h:h + 1, sl].cpu(), dout[b:b + 1, h:h + 1, sl].cpu()
        ks, vs = k[b:b + 1, h:h + 1].cpu(), v[b:b + 1, h:h + 1].cpu()
        rq, _, _ = oracle.attention_bwd(qs, ks, vs, ds, causal=True, scale=w.scale,
                                        query_offset=r0)
        compare_grad(dq[b:b + 1, h:h + 1, sl], rq, f"full-size dQ b={b} h={h} rows {r0}+128")
    dk64 = dk.double()
    dv64 = dv.double()
    sum_dk = dk64.sum(dim=2)                     # [B, H, d]
    sum_dv = dv64.sum(dim=2)
    sum_do = dout.double().sum(dim=2)
    # Each sum adds N bf16-rounded values (relative 2^-9 each, random signs)
    # on top of the per-element error; bound by 1e-2 of the absolute sums.
    abs_dk = dk64.abs().sum(dim=2)
    abs_dv = dv64.abs().sum(dim=2)
    assert (sum_dk.abs() <= 1e-2 * abs_dk + 1e-3).all(), float((sum_dk.abs() / abs_dk).max())
    assert ((sum_dv - sum_do).abs() <= 1e-2 * abs_dv + 1e-3).all(), \
        float(((sum_dv - sum_do).abs() / abs_dv).max())
