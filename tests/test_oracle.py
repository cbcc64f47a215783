"""The fp64 oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.load())


def test_rejects_bad_arguments():
    q = np.zeros((1, 1, 2, 4)); k = np.zeros((1, 1, 3, 4)); v = np.zeros((1, 1, 3, 4))
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, causal=False, scale=1.0, key_range=(2, 1))
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, causal=False, scale=float("nan"))
    with pytest.raises(ValueError):
        oracle.attention(q, np.zeros((1, 1, 3, 5)), v, causal=False, scale=1.0)


def test_bf16_bits_are_widened_exactly():
    """bf16 bit patterns and their float64 values give identical results."""
    import torch
    g = torch.Generator().manual_seed(3)
    q, k, v = (torch.randn((1, 2, n, 16), generator=g).to(torch.bfloat16) for n in (5, 9, 9))
    o1, l1 = oracle.attention(q, k, v, causal=True, scale=0.25)
    o2, l2 = oracle.attention(q.double(), k.double(), v.double(), causal=True, scale=0.25)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_row_subset_matches_full():
    rng = np.random.default_rng(12)
    q = rng.normal(size=(2, 3, 11, 8)); k = rng.normal(size=(2, 3, 14, 8)); v = rng.normal(size=(2, 3, 14, 8))
    o, lse = oracle.attention(q, k, v, causal=True, scale=0.3, query_offset=3)
    rows = np.array([0, 5, 17, 65, 33, 32])
    os_, ls_ = oracle.attention(q, k, v, causal=True, scale=0.3, query_offset=3, rows=rows)
    assert np.array_equal(os_, o.reshape(-1, 8)[rows])
    assert np.array_equal(ls_, lse.reshape(-1)[rows])


def test_thread_count_does_not_change_bits():
    rng = np.random.default_rng(13)
    q = rng.normal(size=(1, 4, 33, 8)); k = rng.normal(size=(1, 4, 40, 8)); v = rng.normal(size=(1, 4, 40, 8))
    a = oracle.attention(q, k, v, causal=False, scale=0.3, threads=1)
    b = oracle.attention(q, k, v, causal=False, scale=0.3, threads=7)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_e4m3_decoder_matches_the_format_and_torch():
    """The oracle's e4m3 decoder: spec values, and torch's converter on all codes."""
    import torch
    from oracle.fp8 import decode_e4m3
    assert decode_e4m3(0x7E) == 448.0          # largest finite
    assert decode_e4m3(0x08) == 2.0 ** -6      # smallest normal
    assert decode_e4m3(0x01) == 2.0 ** -9      # smallest subnormal
    assert decode_e4m3(0x38) == 1.0 and decode_e4m3(0xB8) == -1.0
    assert np.isnan(decode_e4m3(0x7F)) and np.isnan(decode_e4m3(0xFF))
    codes = np.arange(256, dtype=np.uint8)
    ours = decode_e4m3(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    finite = ~np.isnan(ref)
    assert np.array_equal(np.isnan(ours), ~finite)
    assert np.array_equal(ours[finite], ref[finite])


def test_whole_head_chunking_matches_one_call():
    """The chunked evaluation the full-size backward tests use
    (parity_util.whole_head_grads) equals one oracle call on a slice small
    enough to run whole: a check of the tests' own decomposition."""
    from attention_attn_fwd_07_gb300 import inputs as W
    from tests.parity_util import whole_head_grads
    w = W.Workload("chunk check", 1, 2, 300, 300, 64, True, 2700)
    q, k, v = W.make_qkv(w)
    dout = W.make_dout(w)
    rq, rk, rv = oracle.attention_bwd(q[:, 1:2], k[:, 1:2], v[:, 1:2], dout[:, 1:2],
                                      causal=True, scale=w.scale)
    cq, ck, cv = whole_head_grads(oracle, q, k, v, dout, 0, 1, w.scale, chunk=64)
    for a, c in ((rq, cq), (rk, ck), (rv, cv)):
        assert np.allclose(a, c, rtol=1e-12, atol=1e-12)
