"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Every input is seeded and synthetic (attention_attn_fwd_07_gb300.inputs);
the same bf16 bits go to both sides.  Small and ragged cases are compared on
every output element; the full-size workloads, run in the same launch
configuration as the benchmark, are compared on deterministic samples of
rows (tile edges, first/last rows, random rows) that the oracle computes one
by one.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from attention_attn_fwd_07_gb300 import binding, build
from attention_attn_fwd_07_gb300 import inputs as W
from tests.parity_util import check_guards, compare, guarded

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    build.build()
    binding.load_library()
    yield
    assert binding.attn_get_device_status() == 0, "a kernel reported a wait timeout"


def to_dev(*ts):
    return [t.to(DEV) for t in ts]


def oracle_full(q, k, v, causal, scale, query_offset=0):
    return oracle.attention(q, k, v, causal=causal, scale=scale, query_offset=query_offset)


def sample_rows(B, H, Nq, n_heads=8, n_rand=24, seed=0):
    """Flattened row indices: several heads x (edge rows + random rows)."""
    rng = np.random.default_rng(seed)
    BH = B * H
    heads = sorted(set([0, BH - 1] + list(rng.choice(BH, size=min(n_heads, BH), replace=False))))
    edge = [0, 1, 127, 128, 129, 255, 256, 257, Nq // 2, Nq - 2, Nq - 1]
    rows = []
    for h in heads:
        rr = set(i for i in edge if 0 <= i < Nq) | set(rng.integers(0, Nq, size=n_rand).tolist())
        rows += [h * Nq + i for i in sorted(rr)]
    return np.array(rows, dtype=np.int64)


def run_fwd(q, k, v, causal, scale, query_offset=0, flags=0):
    B, H, Nq, d = q.shape
    o, obuf, opad = guarded((B, H, Nq, d), torch.bfloat16, DEV)
    lse, lbuf, lpad = guarded((B, H, Nq), torch.float32, DEV)
    if query_offset == 0 and flags == 0:
        binding.attn_fwd(q, k, v, causal, scale, o=o, lse=lse)
    else:
        binding.attn_fwd_ex(q, k, v, causal, scale, query_offset=query_offset, flags=flags,
                            o=o, lse=lse)
    torch.cuda.synchronize()
    check_guards(obuf, opad, "O")
    check_guards(lbuf, lpad, "LSE")
    return o, lse


def run_split(q, k, v, causal, scale, S, query_offset=0, flags=0):
    B, H, Nq, d = q.shape
    o, obuf, opad = guarded((B, H, Nq, d), torch.bfloat16, DEV)
    lse, lbuf, lpad = guarded((B, H, Nq), torch.float32, DEV)
    need = binding.attn_splitkv_workspace_bytes(B, H, Nq, d, S)
    ws = torch.empty((need + 512,), dtype=torch.uint8, device=DEV)
    ws[need:].fill_(0xA5)
    binding.attn_fwd_splitkv_ex(q, k, v, causal, scale, S, query_offset=query_offset,
                                flags=flags, workspace=ws[:need], o=o, lse=lse)
    torch.cuda.synchronize()
    check_guards(obuf, opad, "O")
    check_guards(lbuf, lpad, "LSE")
    assert (ws[need:].cpu() == 0xA5).all(), "workspace overrun"
    return o, lse


# ------------------------------------------------------------------ small cases
def test_tiny():
    w = W.TINY
    q, k, v = W.make_qkv(w)
    o, lse = run_fwd(*to_dev(q, k, v), w.causal, w.scale)
    compare(o, lse, *oracle_full(q, k, v, w.causal, w.scale), w.name)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", W.RAGGED_LENGTHS)
def test_ragged_fwd(n, causal):
    w = W.ragged(n, causal)
    q, k, v = W.make_qkv(w)
    o, lse = run_fwd(*to_dev(q, k, v), causal, w.scale)
    compare(o, lse, *oracle_full(q, k, v, causal, w.scale), w.name)


@pytest.mark.parametrize("S", W.RAGGED_SPLITS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", W.RAGGED_LENGTHS)
def test_ragged_splitkv(n, causal, S):
    w = W.ragged(n, causal)
    q, k, v = W.make_qkv(w)
    o, lse = run_split(*to_dev(q, k, v), causal, w.scale, S)
    compare(o, lse, *oracle_full(q, k, v, causal, w.scale), f"{w.name} S={S}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_multi_tile_ragged_tail(d, causal):
    """Several 256-row CTA blocks and 128-key tiles with a ragged tail."""
    w = W.Workload("multi-tile", 2, 3, 700, 700, d, causal, 77)
    q, k, v = W.make_qkv(w)
    o, lse = run_fwd(*to_dev(q, k, v), causal, w.scale)
    compare(o, lse, *oracle_full(q, k, v, causal, w.scale), f"d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk,off", [(300, 1000, 700), (129, 520, 3), (1, 1000, 999),
                                       (5, 300, 0), (300, 5, 0)])
def test_query_offset_and_unequal_lengths(d, Nq, Nk, off):
    """Decoding-style subproblems: queries at absolute positions off..off+Nq-1."""
    w = W.Workload("offset", 1, 2, Nq, Nk, d, True, 90 + Nq)
    q, k, v = W.make_qkv(w)
    o, lse = run_fwd(*to_dev(q, k, v), True, w.scale, query_offset=off)
    compare(o, lse, *oracle_full(q, k, v, True, w.scale, off), f"fwd Nq={Nq} Nk={Nk} off={off}")
    for S in (1, 5):
        o, lse = run_split(*to_dev(q, k, v), True, w.scale, S, query_offset=off)
        compare(o, lse, *oracle_full(q, k, v, True, w.scale, off), f"split S={S} off={off}")
    o, lse = run_fwd(*to_dev(q, k, v), False, w.scale)
    compare(o, lse, *oracle_full(q, k, v, False, w.scale), f"fwd non-causal Nq={Nq} Nk={Nk}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("off", [-3, -130, -300])
def test_fully_masked_rows(d, off):
    """Negative query offsets leave leading rows with no admissible key."""
    w = W.Workload("masked", 2, 2, 333, 333, d, True, 55)
    q, k, v = W.make_qkv(w)
    flags = binding.ATTN_FLAG_ALLOW_NEG_OFFSET
    ref = oracle_full(q, k, v, True, w.scale, off)
    assert np.isneginf(ref[1]).any()
    o, lse = run_fwd(*to_dev(q, k, v), True, w.scale, query_offset=off, flags=flags)
    st = compare(o, lse, *ref, f"fwd off={off}")
    assert st["masked_rows"] == 2 * 2 * min(-off, 333)
    for S in (1, 3, 16):
        o, lse = run_split(*to_dev(q, k, v), True, w.scale, S, query_offset=off, flags=flags)
        compare(o, lse, *ref, f"split S={S} off={off}")


def test_single_key_and_causal_row0_are_exact():
    """p = 1 and l = 1 exactly: O is the V row bit for bit, LSE the score."""
    g = torch.Generator().manual_seed(5)
    for d in (64, 128):
        q = torch.randn((2, 2, 37, d), generator=g).bfloat16()
        k = torch.randn((2, 2, 1, d), generator=g).bfloat16()
        v = torch.randn((2, 2, 1, d), generator=g).bfloat16()
        o, lse = run_fwd(*to_dev(q, k, v), False, 0.125)
        assert torch.equal(o.cpu(), v.expand(2, 2, 37, d)), "single key"
        ref = oracle_full(q, k, v, False, 0.125)
        compare(o, lse, *ref, "single key")
        k = torch.randn((2, 2, 37, d), generator=g).bfloat16()
        v = torch.randn((2, 2, 37, d), generator=g).bfloat16()
        o, lse = run_fwd(*to_dev(q, k, v), True, 0.125)
        assert torch.equal(o[:, :, 0].cpu(), v[:, :, 0]), "causal row 0"
        o, lse = run_split(*to_dev(q, k, v), True, 0.125, 4)
        compare(o, lse, *oracle_full(q, k, v, True, 0.125), "split causal")


def test_zero_query_gives_mean_of_v():
    g = torch.Generator().manual_seed(6)
    for d in (64, 128):
        for nk in (1, 200, 1000):
            q = torch.zeros((1, 2, 130, d)).bfloat16()
            k = torch.randn((1, 2, nk, d), generator=g).bfloat16()
            v = torch.randn((1, 2, nk, d), generator=g).bfloat16()
            o, lse = run_fwd(*to_dev(q, k, v), False, 0.125)
            mean = v.double().mean(dim=2, keepdim=True).expand(1, 2, 130, d).numpy()
            compare(o, lse, mean, np.full((1, 2, 130), math.log(nk)), f"q=0 nk={nk}")


def test_constant_v():
    g = torch.Generator().manual_seed(7)
    q = torch.randn((1, 2, 300, 128), generator=g).bfloat16()
    k = (torch.randn((1, 2, 300, 128), generator=g) * 3).bfloat16()
    v = torch.full((1, 2, 300, 128), -1.75).bfloat16()
    for causal in (False, True):
        o, lse = run_fwd(*to_dev(q, k, v), causal, 0.1)
        ref = oracle_full(q, k, v, causal, 0.1)
        compare(o, lse, *ref, "constant V")
        assert np.allclose(o.cpu().double().numpy(), -1.75, atol=1e-2)


@pytest.mark.parametrize("second", [1001.0, 1012.0])
def test_worked_example_large_logits(second):
    """Scores 1000 and `second` in different 128-key tiles (the page's scalar
    example, and a jump large enough to force the O rescale)."""
    g = torch.Generator().manual_seed(8)
    d, nk = 64, 256
    q = torch.zeros((1, 1, 1, d)); q[..., 0] = 1.0; q[..., 1] = 1.0
    k = torch.zeros((1, 1, nk, d)); k[0, 0, 0, 0] = 1000.0
    k[0, 0, 128, 0] = 1000.0; k[0, 0, 128, 1] = second - 1000.0
    v = torch.randn((1, 1, nk, d), generator=g)
    q, k, v = q.bfloat16(), k.bfloat16(), v.bfloat16()
    ref = oracle_full(q, k, v, False, 1.0)
    if second == 1001.0:
        assert abs(ref[1][0, 0, 0] - (1001 + math.log1p(math.exp(-1)))) < 1e-12
    o, lse = run_fwd(*to_dev(q, k, v), False, 1.0)
    compare(o, lse, *ref, f"worked example {second}")
    o, lse = run_split(*to_dev(q, k, v), False, 1.0, 2)
    compare(o, lse, *ref, f"worked example split {second}")


@pytest.mark.parametrize("d", [64, 128])
def test_second_half_spikes(d):
    """Scores that jump in the second half (keys 64-127) of a key tile, on
    the first tile (no O yet) and on a later tile (with an O rescale): the
    maximum of the whole tile must be known before P's first half, which the
    P V product consumes early, is exponentiated."""
    g = torch.Generator().manual_seed(81)
    nk = 256
    q = torch.zeros((1, 1, 4, d))
    for r, a in enumerate((1.0, 0.5, 0.25, -1.0)):
        q[0, 0, r, 0] = a
    k = 0.1 * torch.randn((1, 1, nk, d), generator=g)
    k[0, 0, 0, 0], k[0, 0, 100, 0] = 10.0, 30.0    # tile 0: first half 10, second 30
    k[0, 0, 128, 0], k[0, 0, 200, 0] = 35.0, 60.0  # tile 1: first half 35, second 60
    v = torch.randn((1, 1, nk, d), generator=g)
    q, k, v = q.bfloat16(), k.bfloat16(), v.bfloat16()
    ref = oracle_full(q, k, v, False, 1.0)
    o, lse = run_fwd(*to_dev(q, k, v), False, 1.0)
    compare(o, lse, *ref, f"second-half spikes d={d}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_row_maximum_per_row(d, causal):
    """Each row's exponent reference must be that row's own maximum over the
    whole key tile.  Key j is the unit vector of dimension j mod (d-1) plus a
    shared last dimension; query row i puts 256 on dimension (37 i) mod (d-1)
    and a per-row base in {-256, ..., 256} on the last one, so with scale 1
    row i scores base_i + 256 on one key in each 127 (at a column of the tile
    that moves from row to row) and base_i elsewhere: 369 log2 units apart.
    A reference taken over part of the row overflows 2^x on the hot key; one
    shared across rows (base_i differ by up to 739 log2 units) underflows the
    whole row to zero.  Either leaves O or LSE far from the oracle."""
    nq, nk = 256, 384
    i = torch.arange(nq)
    j = torch.arange(nk)
    q = torch.zeros((1, 1, nq, d))
    q[0, 0, i, (37 * i) % (d - 1)] = 256.0
    q[0, 0, i, d - 1] = 64.0 * ((13 * i) % 9 - 4).float()
    k = torch.zeros((1, 1, nk, d))
    k[0, 0, j, j % (d - 1)] = 1.0
    k[0, 0, :, d - 1] = 1.0
    v = torch.randn((1, 1, nk, d), generator=torch.Generator().manual_seed(82))
    q, k, v = q.bfloat16(), k.bfloat16(), v.bfloat16()
    ref = oracle_full(q, k, v, causal, 1.0)
    o, lse = run_fwd(*to_dev(q, k, v), causal, 1.0)
    compare(o, lse, *ref, f"per-row maximum d={d} causal={causal}")
    o, lse = run_split(*to_dev(q, k, v), causal, 1.0, 3)
    compare(o, lse, *ref, f"per-row maximum split d={d} causal={causal}")


def test_combine_alone():
    """attn_combine on partial states the oracle computes per key range."""
    w = W.Workload("combine", 2, 3, 17, 500, 128, False, 31)
    q, k, v = W.make_qkv(w)
    cuts = [0, 0, 120, 121, 333, 500]  # includes an empty range
    S = len(cuts) - 1
    parts = [oracle.attention(q, k, v, causal=False, scale=w.scale, key_range=(a, b))
             for a, b in zip(cuts[:-1], cuts[1:])]
    o_part = torch.tensor(np.stack([p[0] for p in parts], axis=2), dtype=torch.float32)
    lse_part = torch.tensor(np.stack([p[1] for p in parts], axis=2), dtype=torch.float32)
    o, lse = binding.attn_combine(o_part.to(DEV).contiguous(), lse_part.to(DEV).contiguous(), S)
    torch.cuda.synchronize()
    compare(o, lse, *oracle_full(q, k, v, False, w.scale), "combine")


def test_deterministic():
    w = W.Workload("det", 2, 4, 1000, 1000, 128, True, 44)
    q, k, v = to_dev(*W.make_qkv(w))
    o1, l1 = run_fwd(q, k, v, True, w.scale)
    for _ in range(3):
        o2, l2 = run_fwd(q, k, v, True, w.scale)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    s1 = run_split(q[:, :, :1].contiguous(), k, v, False, w.scale, 7)
    s2 = run_split(q[:, :, :1].contiguous(), k, v, False, w.scale, 7)
    assert torch.equal(s1[0], s2[0]) and torch.equal(s1[1], s2[1])


# ------------------------------------------------------------------ full-size workloads
def _sampled(w, o, lse, q, k, v, rows, query_offset=0, bound=False):
    """Compare the given flattened rows; with ``bound``, also against the
    per-element bound of the bf16 P staging (the oracle run once more with
    |V|)."""
    o_ref, lse_ref = oracle.attention(q, k, v, causal=w.causal, scale=w.scale,
                                      query_offset=query_offset, rows=rows)
    absv = None
    if bound:
        absv, _ = oracle.attention(q, k, v.abs(), causal=w.causal, scale=w.scale,
                                   query_offset=query_offset, rows=rows)
    dv = v.shape[-1]
    o_s = o.reshape(-1, dv)[torch.as_tensor(rows, device=o.device)]
    l_s = lse.reshape(-1)[torch.as_tensor(rows, device=lse.device)]
    return compare(o_s, l_s, o_ref, lse_ref, w.name, absv_ref=absv)


def test_prefill_full_size():
    """Every row of B4 H16 N2048 d64 causal (34 GFLOP for the oracle)."""
    w = W.PREFILL
    q, k, v = W.make_qkv(w)
    o, lse = run_fwd(*to_dev(q, k, v), w.causal, w.scale)
    o_ref, lse_ref = oracle_full(q, k, v, w.causal, w.scale)
    compare(o, lse, o_ref, lse_ref, w.name)


def test_persistent_chunks_straddling_heads():
    """d = 64 causal at B1 H96 N5120: the persistent kernel's causal
    scheduling chunks (on a 152-SM GB300: three of 1216 items and one of
    192, over heads of 40 query blocks) start and end inside heads, and the
    third starts at block 32 of its first head and ends at block 7 of its
    last, so the work-item decode takes every one of its block ranges.  One
    seeded row of every (head, 128-row query block) item, so a missed or
    doubled item shows, plus one whole head."""
    w = W.Workload("chunks B1 H96 N5120 d64 causal", 1, 96, 5120, 5120, 64, True, 1200)
    q, k, v = W.make_qkv(w)
    o, lse = run_fwd(*to_dev(q, k, v), w.causal, w.scale)
    rng = np.random.default_rng(1200)
    n_blocks = w.Nq // 128
    rows = {bh * w.Nq + qb * 128 + int(rng.integers(0, 128))
            for bh in range(w.B * w.H) for qb in range(n_blocks)}
    rows |= set(range(61 * w.Nq, 62 * w.Nq))
    _sampled(w, o, lse, q, k, v, np.array(sorted(rows), dtype=np.int64))


@pytest.mark.parametrize("wl", [W.LONG_PREFILL_CAUSAL, W.LONG_PREFILL_NONCAUSAL],
                         ids=["causal", "noncausal"])
def test_long_prefill_full_size(wl):
    """Two whole (b, h) slices (the last one and one drawn from a seed), every
    row, each element also within the bf16-P bound; plus edge and random rows
    of six more slices."""
    q, k, v = W.make_qkv(wl)
    o, lse = run_fwd(*to_dev(q, k, v), wl.causal, wl.scale)
    BH = wl.B * wl.H
    whole = sorted({BH - 1, int(np.random.default_rng(31).integers(BH - 1))})
    rows = np.concatenate([np.arange(h * wl.Nq, (h + 1) * wl.Nq, dtype=np.int64)
                           for h in whole])
    _sampled(wl, o, lse, q, k, v, rows, bound=True)
    _sampled(wl, o, lse, q, k, v, sample_rows(wl.B, wl.H, wl.Nq, n_heads=6, n_rand=16))


@pytest.fixture(scope="module")
def decode_inputs():
    w = W.DECODE
    q, k, v = W.make_qkv(w, device=DEV)
    return w, q, k, v


@pytest.mark.parametrize("S", W.DECODE.splits)
def test_decode_full_size(decode_inputs, S):
    w, q, k, v = decode_inputs
    o, lse = run_split(q, k, v, w.causal, w.scale, S)
    heads = np.random.default_rng(S).choice(w.B * w.H, size=12, replace=False)
    heads = sorted(set(heads.tolist()) | {0, w.B * w.H - 1})
    idx = torch.as_tensor(heads, device=DEV)
    qh, kh, vh = (t.reshape(w.B * w.H, -1, w.d)[idx].unsqueeze(0).cpu() for t in (q, k, v))
    o_ref, lse_ref = oracle.attention(qh, kh, vh, causal=w.causal, scale=w.scale)
    compare(o.reshape(w.B * w.H, 1, w.d)[idx].unsqueeze(0), lse.reshape(w.B * w.H, 1)[idx].unsqueeze(0),
            o_ref, lse_ref, f"decode S={S}")
