"""The pinned-host-buffer entry (fwd_from_host) pipelines chunks of heads
over an upload stream, the compute stream and a download stream: the result
in the host buffers must equal the oracle's, for chunk sizes that do and do
not divide the head count, with grouped K/V heads, and must not depend on
the chunking."""
import pytest
import torch

import oracle
from attention_attn_fwd_07_gb300 import binding, build
from attention_attn_fwd_07_gb300 import inputs as W
from tests.parity_util import compare

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    build.build()
    binding.load_library()


def run(w, chunk_heads, causal=True):
    q, k, v = W.make_qkv(w)
    qp, kp, vp = (t.pin_memory() for t in (q, k, v))
    qd, kd, vd = torch.empty_like(q, device=DEV), torch.empty_like(k, device=DEV), torch.empty_like(v, device=DEV)
    od = torch.empty_like(qd)
    ld = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=DEV)
    op = torch.full(q.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    lp = torch.full((w.B, w.H, w.Nq), float("nan"), dtype=torch.float32).pin_memory()
    s = torch.cuda.Stream()
    binding.fwd_from_host(qp, kp, vp, causal, w.scale, qd, kd, vd, od, ld, op, lp, stream=s,
                          chunk_heads=chunk_heads)
    s.synchronize()
    return q, k, v, op, lp


@pytest.mark.parametrize("chunk_heads", [1, 3, 8, 64])
def test_from_host_matches_oracle(chunk_heads):
    w = W.Workload("from host", 2, 6, 300, 300, 128, True, 4000)
    q, k, v, op, lp = run(w, chunk_heads)
    compare(op, lp, *oracle.attention(q, k, v, causal=True, scale=w.scale),
            f"from host chunk_heads={chunk_heads}")


def test_from_host_grouped_heads_and_chunking_invariance():
    w = W.Workload("from host gqa", 2, 8, 257, 257, 64, True, 4001, Hkv=2)
    q, k, v, o1, l1 = run(w, 4)
    _, _, _, o2, l2 = run(w, 8)
    compare(o1, l1, *oracle.attention(q, k, v, causal=True, scale=w.scale), "from host gqa")
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)
