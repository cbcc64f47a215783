"""attn_fwd_splitkv_noalloc against attn_fwd_splitkv, through the C ABI.

The allocation-free entry point exists for callers that cannot allocate
device memory: code whose device memory is all planned by an outer arena that
refuses further allocation, plug-ins whose host program exposes no
allocator, and latency-critical loops that cannot afford the device
synchronisation cudaMalloc/cudaFree may cause.  It keeps the split-KV
scratch in a fixed 32 MiB array inside the library instead of a caller
workspace.  Here it must meet the fp64 oracle within the parity tolerances,
as the workspace entry point does (the two may run different partial kernels
for the same shape, so they are each compared with the oracle, not
bitwise), on problems called one after the other, and must refuse a problem
whose scratch exceeds the array.

The outputs of the two entry points are also compared with each other
within the same tolerances.  One case fills the array almost to its end (its
partial log-sum-exps sit in the last few hundred KiB), and the same shape
with more splits must be refused.

This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from attention_attn_fwd_07_gb300 import binding, build
from attention_attn_fwd_07_gb300 import inputs as W
from tests.parity_util import LSE_TOL, O_TOL, compare, half_ulp_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SCRATCH_BYTES = 32 << 20  # ATTN_NOALLOC_SCRATCH_BYTES in include/attn.h


def _agree(o_a, lse_a, o_b, lse_b, what):
    """The two entry points' outputs within the parity tolerances: LSE within
    1e-3 (-inf rows exactly alike); O within 1e-2 beyond the two outputs' own
    bf16 roundings (half an ulp each), the rule the oracle comparison applies
    to one output."""
    la, lb = lse_a.double().cpu(), lse_b.double().cpu()
    assert torch.equal(torch.isneginf(la), torch.isneginf(lb)), f"{what}: masked rows differ"
    live = ~torch.isneginf(la)
    assert (la[live] - lb[live]).abs().max().item() <= LSE_TOL, f"{what}: LSE differs"
    a, b = o_a.double().cpu().numpy(), o_b.double().cpu().numpy()
    excess = np.abs(a - b) - half_ulp_bf16(a) - half_ulp_bf16(b)
    assert excess.max() <= O_TOL, f"{what}: O differs by {excess.max()} beyond rounding"


def _entry(lib):
    f = lib.attn_fwd_splitkv_noalloc
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    f.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_float,
                  ctypes.c_int, vp]
    f.restype = ctypes.c_int
    return f


def _call(f, q, k, v, o, lse, causal, scale, splits):
    B, H, Nq, d = q.shape
    return f(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Nq,
             k.shape[2], d, int(causal), float(scale), int(splits),
             torch.cuda.current_stream().cuda_stream)


def test_noalloc_parity_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    build.build()
    f = _entry(binding.load_library())
    cases = [(W.Workload("decode-like", 2, 8, 1, 5000, 128, False, 501), 8),
             (W.Workload("short causal queries", 3, 2, 37, 777, 64, True, 502), 5),
             # several rows per head at d = 128: the pipelined CUDA-core kernel
             (W.Workload("short causal queries d128", 2, 4, 5, 900, 128, True, 503), 4)]
    for w, splits in cases:
        q_h, k_h, v_h = W.make_qkv(w)
        q, k, v = (t.to(DEV) for t in (q_h, k_h, v_h))
        ref = oracle.attention(q_h, k_h, v_h, causal=w.causal, scale=w.scale)
        o_ws, lse_ws = binding.attn_fwd_splitkv(q, k, v, w.causal, w.scale, splits)
        o = torch.full_like(o_ws, float("nan"))
        lse = torch.full_like(lse_ws, float("nan"))
        assert _call(f, q, k, v, o, lse, w.causal, w.scale, splits) == binding.ATTN_OK
        torch.cuda.synchronize()
        compare(o, lse, *ref, f"{w.name} (no-alloc entry point)")
        compare(o_ws, lse_ws, *ref, f"{w.name} (workspace entry point)")
        _agree(o, lse, o_ws, lse_ws, w.name)


def test_noalloc_fills_the_array_to_its_end():
    """B16 H32 Nq1 d128 with 127 splits needs all but 2 KiB of the 32 MiB
    array, so the partial log-sum-exps occupy its last 254 KiB; with
    Nk = 2000 only 16 of the 127 key ranges hold keys and the rest are empty
    (o = 0, lse = -inf partials).  Two calls in a row must both match the
    oracle, and 128 splits at the same shape must be refused."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    build.build()
    f = _entry(binding.load_library())
    w = W.Workload("near the end of the array", 16, 32, 1, 2000, 128, False, 504)
    splits = 127
    need = binding.attn_splitkv_workspace_bytes(w.B, w.H, 1, w.d, splits)
    assert SCRATCH_BYTES - 4096 < need <= SCRATCH_BYTES
    q_h, k_h, v_h = W.make_qkv(w)
    q, k, v = (t.to(DEV) for t in (q_h, k_h, v_h))
    ref = oracle.attention(q_h, k_h, v_h, causal=False, scale=w.scale)
    o_ws, lse_ws = binding.attn_fwd_splitkv(q, k, v, False, w.scale, splits)
    for call in range(2):
        o = torch.full_like(o_ws, float("nan"))
        lse = torch.full_like(lse_ws, float("nan"))
        assert _call(f, q, k, v, o, lse, False, w.scale, splits) == binding.ATTN_OK
        torch.cuda.synchronize()
        compare(o, lse, *ref, f"{w.name}, call {call + 1}")
        _agree(o, lse, o_ws, lse_ws, f"{w.name}, call {call + 1}")
    assert binding.attn_splitkv_workspace_bytes(w.B, w.H, 1, w.d, 128) > SCRATCH_BYTES
    assert _call(f, q, k, v, o, lse, False, w.scale, 128) == binding.ATTN_ERR_WORKSPACE


def test_noalloc_refuses_scratch_beyond_its_array():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    build.build()
    f = _entry(binding.load_library())
    B, H, d, splits = 16, 32, 128, 256
    assert binding.attn_splitkv_workspace_bytes(B, H, 1, d, splits) > SCRATCH_BYTES
    q = torch.zeros((B, H, 1, d), dtype=torch.bfloat16, device=DEV)
    o = torch.zeros_like(q)
    lse = torch.zeros((B, H, 1), dtype=torch.float32, device=DEV)
    assert _call(f, q, q, q, o, lse, False, 0.125, splits) == binding.ATTN_ERR_WORKSPACE
