"""Pins that tie the fp64 oracle to what the pages and mathematics fix.

Each ``pin_*`` takes an oracle library handle (the real one, or a variant
built with a planted mistake) and raises AssertionError when the property
fails.  ``tests/test_oracle.py`` runs them on the real oracle;
``tests/test_oracle_plants.py`` shows that every planted mistake trips at
least one of them.

Sources ("GPU Engineering: Correctness, Throughput, and Attention"):
  * section 22.5: the online recurrence (m, l, o) with rescaling by
    alpha = exp(m - m_new) reaches the full stable softmax; causal masking is
    applied before maxima and sums; fully masked rows need explicit semantics.
  * section 22.7: the scalar example with scores 1000 and 1001 in separate
    tiles; the lab's causal rule (key j excluded when j > i + query_offset),
    its zero-output / -inf log-normaliser policy, its natural-log
    log-normaliser m + ln(l), and its tile sizes 1, 4 and > keys that must
    agree within rounding.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
RTOL = 1e-12


def _att(lib, q, k, v, causal, scale, offset=0, key_range=None, rows=None):
    return oracle.attention(q, k, v, causal=causal, scale=scale, query_offset=offset,
                            key_range=key_range, rows=rows, threads=2, lib=lib)


def _bf16_like(rng, shape, scale=1.0):
    """float64 values that are exactly representable in bfloat16."""
    x = rng.normal(size=shape) * scale
    bits = x.astype(np.float32).view(np.uint32)
    bits = (bits + 0x7FFF + ((bits >> 16) & 1)) & 0xFFFF0000  # round to nearest even
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)


def _close(a, b, rtol=RTOL, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    same_inf = (np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b)))
    fin = ~same_inf
    assert not np.isnan(a).any(), f"{what}: NaN in oracle output"
    err = np.abs(a[fin] - b[fin])
    tol = rtol * np.maximum(1.0, np.abs(b[fin]))
    assert (err <= tol).all(), f"{what}: max err {err.max() if err.size else 0:.3e}"
    assert (np.isinf(a) == np.isinf(b)).all(), f"{what}: infinities differ"


def online_reference(q, k, v, tile, causal, scale, offset):
    """Test-only restatement of the section 22.5 recurrence for one head.

    q: [Nq, d], k: [Nk, d], v: [Nk, dv], float64.  Keys are visited in tiles
    of ``tile``; a still-fully-masked row uses 0 as its exponent reference.
    """
    Nq, Nk = q.shape[0], k.shape[0]
    m = np.full(Nq, -np.inf)
    l = np.zeros(Nq)
    o = np.zeros((Nq, v.shape[1]))
    for start in range(0, Nk, tile):
        kt, vt = k[start:start + tile], v[start:start + tile]
        s = (q @ kt.T) * scale
        if causal:
            keys = np.arange(start, start + len(kt))[None, :]
            rows = np.arange(Nq)[:, None] + offset
            s = np.where(keys > rows, -np.inf, s)
        m_new = np.maximum(m, s.max(axis=1))
        ref = np.where(np.isfinite(m_new), m_new, 0.0)
        alpha = np.exp(m - ref)
        p = np.exp(s - ref[:, None])
        o = alpha[:, None] * o + p @ vt
        l = alpha * l + p.sum(axis=1)
        m = m_new
    out = np.zeros_like(o)
    nz = l > 0
    out[nz] = o[nz] / l[nz, None]
    lse = np.full(Nq, -np.inf)
    lse[nz] = m[nz] + np.log(l[nz])
    return out, lse


def pin_online_matches_two_pass(lib):
    """Tiled online softmax (tiles 1, 4, > Nk) equals the dense oracle."""
    rng = np.random.default_rng(0)
    # The lab's demo shapes: Q 7x5, K 11x5, V 11x3, causal.
    q, k, v = (rng.normal(size=s) for s in ((7, 5), (11, 5), (11, 3)))
    cases = [(q, k, v, True, 0), (q, k, v, False, 0), (q, k, v, True, 3)]
    rng2 = np.random.default_rng(7)
    q2 = _bf16_like(rng2, (37, 16))
    k2 = _bf16_like(rng2, (45, 16), scale=2.0)
    v2 = _bf16_like(rng2, (45, 16))
    cases += [(q2, k2, v2, True, 8), (q2, k2, v2, False, 0)]
    for q, k, v, causal, off in cases:
        scale = 1.0 / math.sqrt(q.shape[1])
        o_ref, lse_ref = _att(lib, q[None, None], k[None, None], v[None, None], causal,
                              scale, off)
        for tile in (1, 4, k.shape[0] + 5):
            o_t, lse_t = online_reference(q, k, v, tile, causal, scale, off)
            _close(o_ref[0, 0], o_t, what=f"O tile={tile} causal={causal} off={off}")
            _close(lse_ref[0, 0], lse_t, what=f"LSE tile={tile} causal={causal} off={off}")


def _scores(q, k, causal, scale, offset):
    s = np.einsum("bhid,bhjd->bhij", q, k) * scale
    if causal:
        i = np.arange(q.shape[2])[:, None] + offset
        j = np.arange(k.shape[2])[None, :]
        s = np.where(j > i, -np.inf, s)
    return s


def pin_rows_sum_to_one(lib):
    """sum_j exp(s_j - LSE) = 1 for every row with an admissible key."""
    rng = np.random.default_rng(1)
    q = _bf16_like(rng, (2, 3, 19, 8))
    k = _bf16_like(rng, (2, 3, 23, 8), scale=3.0)
    v = _bf16_like(rng, (2, 3, 23, 8))
    for causal in (False, True):
        _, lse = _att(lib, q, k, v, causal, 0.35)
        s = _scores(q, k, causal, 0.35, 0)
        total = np.exp(s - lse[..., None]).sum(axis=-1)
        assert np.all(np.abs(total - 1.0) <= 1e-12), f"row sums off by {np.abs(total - 1).max()}"


def pin_single_key(lib):
    """One key returns its V row exactly and LSE equals its score exactly."""
    rng = np.random.default_rng(2)
    q = _bf16_like(rng, (1, 2, 5, 16))
    k = _bf16_like(rng, (1, 2, 1, 16))
    v = _bf16_like(rng, (1, 2, 1, 16))
    o, lse = _att(lib, q, k, v, False, 0.25)
    assert np.array_equal(o, np.broadcast_to(v, o.shape)), "single key: O != V row"
    exact = np.einsum("bhid,bhjd->bhij", q, k)[..., 0] * 0.25
    assert np.array_equal(lse, exact), "single key: LSE != score"
    # Causal row 0 sees key 0 only.
    q = _bf16_like(rng, (1, 2, 9, 16))
    k = _bf16_like(rng, (1, 2, 9, 16))
    v = _bf16_like(rng, (1, 2, 9, 16))
    o, lse = _att(lib, q, k, v, True, 0.25)
    assert np.array_equal(o[:, :, 0], v[:, :, 0]), "causal row 0: O != V[0]"
    exact0 = (q[:, :, 0] * k[:, :, 0]).sum(-1) * 0.25
    assert np.array_equal(lse[:, :, 0], exact0), "causal row 0: LSE != s_00"


def pin_zero_query(lib):
    """q = 0 makes every score 0: O = mean(V), LSE = ln(Nk)."""
    rng = np.random.default_rng(3)
    for nk in (1, 6, 33):
        q = np.zeros((1, 1, 4, 8))
        k = _bf16_like(rng, (1, 1, nk, 8))
        v = _bf16_like(rng, (1, 1, nk, 8))
        o, lse = _att(lib, q, k, v, False, 0.5)
        _close(o[0, 0], np.broadcast_to(v[0, 0].mean(axis=0), (4, 8)), 1e-14, "mean V")
        _close(lse, np.full((1, 1, 4), math.log(nk)), 1e-14, "ln Nk")


def pin_constant_v(lib):
    """Constant V = c gives O = c in every row with an admissible key."""
    rng = np.random.default_rng(4)
    q = _bf16_like(rng, (2, 1, 10, 8))
    k = _bf16_like(rng, (2, 1, 12, 8), scale=4.0)
    v = np.full((2, 1, 12, 8), -1.75)
    for causal in (False, True):
        o, _ = _att(lib, q, k, v, causal, 0.5)
        _close(o, np.full_like(o, -1.75), 1e-14, "constant V")


def pin_worked_example(lib):
    """Section 22.7's scalar example, alone and embedded at d = 64."""
    with open(os.path.join(GOLDEN, "online_softmax_scalar_example.json")) as f:
        g = json.load(f)
    m2 = g["after_tile_2"]["m"]
    l2 = g["after_tile_2"]["l"]
    rescale = g["rescale_of_first_contribution"]
    assert abs(l2 - (math.exp(-1) + 1)) < 1e-15 and abs(rescale - math.exp(-1)) < 1e-15
    lse_expected = m2 + math.log(l2)  # the lab's log-normaliser: maximum + ln(normaliser)

    # Scalar form: d = 1, q = 1, keys 1000 and 1001, scale 1.
    v = np.array([[[[2.0], [-3.0]]]])
    o, lse = _att(lib, np.ones((1, 1, 1, 1)),
                  np.array(g["scores"]).reshape(1, 1, 2, 1), v, False, 1.0)
    _close(lse[0, 0, 0], lse_expected, 1e-15, "scalar LSE")
    _close(o[0, 0, 0, 0], (rescale * 2.0 + 1.0 * -3.0) / l2, 1e-14, "scalar O")

    # Embedded: d = 64, keys 0 and 128 score 1000 and 1001, the rest score 0.
    rng = np.random.default_rng(5)
    d, nk = 64, 256
    q = np.zeros((1, 1, 1, d)); q[..., 0] = 1.0; q[..., 1] = 1.0
    k = np.zeros((1, 1, nk, d)); k[0, 0, 0, 0] = 1000.0
    k[0, 0, 128, 0] = 1000.0; k[0, 0, 128, 1] = 1.0
    v = _bf16_like(rng, (1, 1, nk, d))
    o, lse = _att(lib, q, k, v, False, 1.0)
    _close(lse[0, 0, 0], lse_expected, 1e-15, "embedded LSE")
    o_expected = (rescale * v[0, 0, 0] + v[0, 0, 128]) / l2
    _close(o[0, 0, 0], o_expected, 1e-14, "embedded O")


def brute_force(q, k, v, causal, scale, offset):
    """Pure-Python triple loop with exactly rounded sums (math.fsum)."""
    Nq, Nk, dv = len(q), len(k), len(v[0])
    out, lse = [], []
    for i in range(Nq):
        s = []
        for j in range(Nk):
            if causal and j > i + offset:
                s.append(None)
            else:
                s.append(math.fsum(q[i][c] * k[j][c] for c in range(len(q[i]))) * scale)
        live = [x for x in s if x is not None]
        if not live:
            out.append([0.0] * dv)
            lse.append(-math.inf)
            continue
        mx = max(live)
        w = [0.0 if x is None else math.exp(x - mx) for x in s]
        z = math.fsum(w)
        out.append([math.fsum(w[j] * v[j][c] for j in range(Nk)) / z for c in range(dv)])
        lse.append(mx + math.log(z))
    return out, lse


def pin_brute_force(lib):
    """Oracle equals an independent pure-Python evaluation on tiny inputs."""
    rng = np.random.default_rng(0)
    q, k, v = (rng.normal(size=s) for s in ((7, 5), (11, 5), (11, 3)))
    cases = [(q, k, v, True, 0, 1 / math.sqrt(5)), (q, k, v, False, 0, 1 / math.sqrt(5)),
             (q, k, v, True, -3, 0.7)]
    rng = np.random.default_rng(11)
    q2 = _bf16_like(rng, (9, 4)); k2 = _bf16_like(rng, (6, 4), 3.0); v2 = _bf16_like(rng, (6, 4))
    cases += [(q2, k2, v2, True, 2, 0.5), (q2, k2, v2, False, 0, 1.5)]
    for q, k, v, causal, off, scale in cases:
        o, lse = _att(lib, q[None, None], k[None, None], v[None, None], causal, scale, off)
        o_b, lse_b = brute_force(q.tolist(), k.tolist(), v.tolist(), causal, scale, off)
        _close(o[0, 0], np.array(o_b), 1e-13, f"brute O causal={causal} off={off}")
        _close(lse[0, 0], np.array(lse_b), 1e-13, f"brute LSE causal={causal} off={off}")


def pin_fully_masked_policy(lib):
    """Rows with no admissible key: O exactly +0.0, LSE exactly -inf, no NaN."""
    rng = np.random.default_rng(6)
    q = _bf16_like(rng, (1, 2, 8, 8)); k = _bf16_like(rng, (1, 2, 8, 8)); v = _bf16_like(rng, (1, 2, 8, 8))
    o, lse = _att(lib, q, k, v, True, 0.5, offset=-3)
    assert np.all(o[:, :, :3] == 0.0) and not np.signbit(o[:, :, :3]).any(), "masked O"
    assert np.all(np.isneginf(lse[:, :, :3])), "masked LSE"
    assert np.all(np.isfinite(lse[:, :, 3:])), "row 3 onward must see keys"
    o_empty, lse_empty = _att(lib, q, k, v, False, 0.5, key_range=(4, 4))
    assert np.all(o_empty == 0.0) and np.all(np.isneginf(lse_empty)), "empty key range"


def pin_permutation_invariance(lib):
    """Non-causal: permuting K and V rows together changes nothing."""
    rng = np.random.default_rng(8)
    q = _bf16_like(rng, (2, 2, 7, 8)); k = _bf16_like(rng, (2, 2, 29, 8), 2.0)
    v = _bf16_like(rng, (2, 2, 29, 8))
    perm = rng.permutation(29)
    o1, l1 = _att(lib, q, k, v, False, 0.4)
    o2, l2 = _att(lib, q, k[:, :, perm], v[:, :, perm], False, 0.4)
    _close(o1, o2, 1e-12, "perm O")
    _close(l1, l2, 1e-12, "perm LSE")


def pin_shift_invariance(lib):
    """Adding t*q to every key shifts one row's scores by a constant."""
    rng = np.random.default_rng(9)
    q = _bf16_like(rng, (1, 1, 1, 8)); k = _bf16_like(rng, (1, 1, 17, 8))
    v = _bf16_like(rng, (1, 1, 17, 8))
    t, scale = 0.75, 0.3
    o1, l1 = _att(lib, q, k, v, False, scale)
    o2, l2 = _att(lib, q, k + t * q, v, False, scale)
    shift = t * float((q * q).sum()) * scale
    _close(o2, o1, 1e-12, "shift O")
    _close(l2, l1 + shift, 1e-12, "shift LSE")


def merge(parts):
    """Merge per-key-range (o, lse) pairs by log-sum-exp weights."""
    lses = np.stack([p[1] for p in parts])
    m = lses.max(axis=0)
    safe = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lses - safe)
    z = w.sum(axis=0)
    o = sum(wi[..., None] * p[0] for wi, p in zip(w, parts))
    out = np.where(z[..., None] > 0, o / np.where(z > 0, z, 1)[..., None], 0.0)
    lse = np.where(z > 0, safe + np.log(np.where(z > 0, z, 1)), -np.inf)
    return out, lse


def pin_split_merge(lib):
    """Attention over disjoint key ranges, merged by LSE, equals the full one."""
    rng = np.random.default_rng(10)
    q = _bf16_like(rng, (1, 2, 13, 8)); k = _bf16_like(rng, (1, 2, 40, 8), 2.0)
    v = _bf16_like(rng, (1, 2, 40, 8))
    for causal in (False, True):
        full = _att(lib, q, k, v, causal, 0.5)
        for cuts in ((0, 13, 40), (0, 0, 7, 7, 31, 40), (0, 40, 40)):
            parts = [_att(lib, q, k, v, causal, 0.5, key_range=(a, b))
                     for a, b in zip(cuts[:-1], cuts[1:])]
            o, lse = merge(parts)
            _close(o, full[0], 1e-12, f"merge O {cuts}")
            _close(lse, full[1], 1e-12, f"merge LSE {cuts}")


def pin_grouped_heads_equal_replicated_heads(lib):
    """GQA/MQA: K/V heads shared by groups of query heads give exactly the
    result of multi-head attention with each K/V head repeated for its group."""
    rng = np.random.default_rng(14)
    B, H, Nq, Nk, d = 2, 6, 9, 13, 8
    q = _bf16_like(rng, (B, H, Nq, d))
    for hkv in (1, 2, 3, 6):
        k = _bf16_like(rng, (B, hkv, Nk, d), 2.0)
        v = _bf16_like(rng, (B, hkv, Nk, d))
        kr = np.repeat(k, H // hkv, axis=1)
        vr = np.repeat(v, H // hkv, axis=1)
        for causal in (False, True):
            o1, l1 = _att(lib, q, k, v, causal, 0.4, offset=2)
            o2, l2 = _att(lib, q, kr, vr, causal, 0.4, offset=2)
            assert np.array_equal(o1, o2) and np.array_equal(l1, l2), f"Hkv={hkv}"


def _bwd(lib, q, k, v, g, causal, scale, offset=0):
    return oracle.attention_bwd(q, k, v, g, causal=causal, scale=scale, query_offset=offset,
                                threads=2, lib=lib)


def pin_bwd_finite_differences(lib):
    """Gradients against central finite differences of L = sum(O * G) in fp64
    (the lab's check: perturb Q, K, V separately in random directions)."""
    rng = np.random.default_rng(21)
    cases = []
    q, k, v = (rng.normal(size=s)[None, None] for s in ((7, 5), (11, 5), (11, 5)))
    cases += [(q, k, v, True, 0), (q, k, v, True, 2), (q, k, v, False, 0)]
    q = rng.normal(size=(1, 4, 6, 4)); k = rng.normal(size=(1, 2, 9, 4))
    v = rng.normal(size=(1, 2, 9, 4))
    cases += [(q, k, v, False, 0), (q, k, v, True, 3)]
    # value width different from the key width (dv 3 and 7 against d 5)
    q, k = (rng.normal(size=s)[None, None] for s in ((7, 5), (11, 5)))
    for e in (3, 7):
        v = rng.normal(size=(11, e))[None, None]
        cases += [(q, k, v, True, 1), (q, k, v, False, 0)]
    eps = 1e-5
    for q, k, v, causal, off in cases:
        scale = 0.6
        g = rng.normal(size=q.shape[:3] + v.shape[3:])
        dq, dk, dv = _bwd(lib, q, k, v, g, causal, scale, off)

        def loss(qq, kk, vv):
            o, _ = _att(lib, qq, kk, vv, causal, scale, off)
            return float((o * g).sum())

        for name, x, dx in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            u = rng.normal(size=x.shape)
            args_p = [q, k, v]; args_m = [q, k, v]
            i = "qkv".index(name)
            args_p[i] = x + eps * u
            args_m[i] = x - eps * u
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            an = float((dx * u).sum())
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), f"d{name}: fd {fd} vs {an}"


def backward_reference(q, k, v, g, o, lse, tile, causal, scale, offset):
    """Test-only restatement of the lab's recomputing backward for one head:
    P recomputed tile by tile as exp(scores - LSE), row correction
    rowsum(G * O); q, g [Nq, d], k, v [Nk, d]."""
    Nq, Nk = q.shape[0], k.shape[0]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    corr = (g * o).sum(axis=1)
    valid = np.isfinite(lse)
    ref = np.where(valid, lse, 0.0)
    for start in range(0, Nk, tile):
        kt, vt = k[start:start + tile], v[start:start + tile]
        s = (q @ kt.T) * scale
        if causal:
            keys = np.arange(start, start + len(kt))[None, :]
            s = np.where(keys > np.arange(Nq)[:, None] + offset, -np.inf, s)
        p = np.exp(s - ref[:, None])
        p[~valid] = 0.0
        ds = p * (g @ vt.T - corr[:, None])
        dq += (ds @ kt) * scale
        dk[start:start + tile] += (ds.T @ q) * scale
        dv[start:start + tile] += p.T @ g
    return dq, dk, dv


def pin_bwd_tiled_recompute(lib):
    """The lab's tiled backward (tiles 1, 4, > Nk, recompute from LSE, row
    correction rowsum(dO * O)) equals the dense definition."""
    rng = np.random.default_rng(22)
    q, k, v = (_bf16_like(rng, s) for s in ((9, 8), (13, 8), (13, 8)))
    g = _bf16_like(rng, (9, 8))
    for causal, off in ((True, 0), (True, 4), (False, 0), (True, -3)):
        o, lse = _att(lib, q[None, None], k[None, None], v[None, None], causal, 0.45, off)
        ref = _bwd(lib, q[None, None], k[None, None], v[None, None], g[None, None], causal,
                   0.45, off)
        for tile in (1, 4, 20):
            mine = backward_reference(q, k, v, g, o[0, 0], lse[0, 0], tile, causal, 0.45, off)
            for name, a, b in zip("qkv", ref, mine):
                _close(a[0, 0], b, 1e-11, f"d{name} tile={tile} causal={causal} off={off}")


def pin_bwd_single_key(lib):
    """One key: P = 1, so dS = 0 (dQ = dK = 0 exactly) and dV = sum of dO."""
    rng = np.random.default_rng(23)
    q = _bf16_like(rng, (2, 4, 5, 8)); k = _bf16_like(rng, (2, 2, 1, 8))
    v = _bf16_like(rng, (2, 2, 1, 8)); g = _bf16_like(rng, (2, 4, 5, 8))
    dq, dk, dv = _bwd(lib, q, k, v, g, False, 0.3)
    assert np.array_equal(dq, np.zeros_like(dq)) and np.array_equal(dk, np.zeros_like(dk))
    expect = g.reshape(2, 2, 2 * 5, 8).sum(axis=2, keepdims=True)
    _close(dv, expect, 1e-15, "single key dV")


def pin_bwd_masked_rows_and_keys(lib):
    """Rows without admissible keys get zero dQ; keys no row can see get zero
    dK and dV (exact zeros)."""
    rng = np.random.default_rng(24)
    q = _bf16_like(rng, (1, 2, 6, 8)); k = _bf16_like(rng, (1, 2, 10, 8))
    v = _bf16_like(rng, (1, 2, 10, 8)); g = _bf16_like(rng, (1, 2, 6, 8))
    dq, dk, dv = _bwd(lib, q, k, v, g, True, 0.5, offset=-2)
    assert np.all(dq[:, :, :2] == 0.0) and np.any(dq[:, :, 2:] != 0.0)
    # rows 0..5 with offset -2 see keys <= 3; keys 4..9 are never attended
    assert np.all(dk[:, :, 4:] == 0.0) and np.all(dv[:, :, 4:] == 0.0)
    assert np.any(dk[:, :, :4] != 0.0) and np.any(dv[:, :, :4] != 0.0)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
