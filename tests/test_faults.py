"""Failure detection without a GPU fault: the prefill kernel's bounded waits.

ATTN_FLAG_TEST_SKIP_LOAD makes the kernel's TMA producer skip one V tile, so
the MMA warp's wait for it can never complete.  With a short per-wait limit
the kernel must record ATTN_ERR_DEVICE_TIMEOUT in the status word, leave the
pipeline (awaiting its own copies and MMAs in flight), free its tensor
memory and return; the context stays usable and the next normal call is
exact again.  No trap, assert or bad address is involved.
"""
import pytest
import torch

import oracle
from attention_attn_fwd_07_gb300 import binding, build
from attention_attn_fwd_07_gb300 import inputs as W
from tests.parity_util import compare

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TIMEOUT_US = 20000  # 20 ms per wait; a handful of CTAs, so the call ends in well under a second


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    build.build()
    binding.load_library()
    binding.attn_get_device_status()  # start from a clear status word


@pytest.mark.parametrize("d", [64, 128])
def test_skipped_load_times_out_and_context_survives(d):
    w = W.Workload("fault", 1, 2, 600, 600, d, True, 71)
    q, k, v = W.make_qkv(w)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))

    binding.attn_fwd_ex(qd, kd, vd, True, w.scale, flags=binding.ATTN_FLAG_TEST_SKIP_LOAD,
                        wait_timeout_us=TIMEOUT_US)
    status = binding.attn_get_device_status()
    assert status & 1, "the skipped load must surface as a device timeout"
    assert binding.attn_get_device_status() == 0, "reading the status word clears it"

    o, lse = binding.attn_fwd(qd, kd, vd, True, w.scale)
    torch.cuda.synchronize()
    compare(o, lse, *oracle.attention(q, k, v, causal=True, scale=w.scale), "after timeout")
    assert binding.attn_get_device_status() == 0


def test_timeout_goes_to_the_callers_status_word():
    w = W.Workload("fault", 1, 1, 300, 300, 128, False, 72)
    qd, kd, vd = (t.to(DEV) for t in W.make_qkv(w))
    mine = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.attn_fwd_ex(qd, kd, vd, False, w.scale, flags=binding.ATTN_FLAG_TEST_SKIP_LOAD,
                        dev_status=mine, wait_timeout_us=TIMEOUT_US)
    torch.cuda.synchronize()
    assert int(mine.item()) & 1
    assert binding.attn_get_device_status() == 0, "the library's own word stays clear"
