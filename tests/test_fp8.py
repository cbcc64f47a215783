"""GPU parity for FP8 Q K^T (e4m3 Q and K with per-tensor descales, bf16 V):
the prefill kernel's kind::f8f6f4 path against the fp64 oracle on the same
e4m3 codes, decoded exactly; scores are scale * q_descale * k_descale * <q,k>."""
import numpy as np
import pytest
import torch

import oracle
from oracle.fp8 import decode_e4m3
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
    assert binding.attn_get_device_status() == 0


def oracle_inputs(q8, k8, v):
    return decode_e4m3(q8.numpy()), decode_e4m3(k8.numpy()), v.double().numpy()


def run_fp8(q8, k8, v, causal, scale, qd, kd, query_offset=0):
    B, H, Nq, d = q8.shape
    o, obuf, opad = guarded((B, H, Nq, v.shape[3]), torch.bfloat16, DEV)
    lse, lbuf, lpad = guarded((B, H, Nq), torch.float32, DEV)
    binding.attn_fwd_fp8(q8.to(DEV), k8.to(DEV), v.to(DEV), causal, scale, qd, kd,
                         query_offset=query_offset, o=o, lse=lse)
    torch.cuda.synchronize()
    check_guards(obuf, opad, "O")
    check_guards(lbuf, lpad, "LSE")
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,hkv", [(1, 2), (128, 2), (333, 2), (700, 1), (1003, 2)])
def test_fp8_prefill(n, hkv, causal):
    w = W.Workload("fp8", 2, 2, n, n, 128, causal, 500 + n, Hkv=hkv)
    q8, k8, v, qd, kd = W.make_qkv_fp8(w)
    o, lse = run_fp8(q8, k8, v, causal, w.scale, qd, kd)
    qo, ko, vo = oracle_inputs(q8, k8, v)
    ref = oracle.attention(qo, ko, vo, causal=causal, scale=w.scale * qd * kd)
    compare(o, lse, *ref, f"fp8 n={n} Hkv={hkv} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", [129, 1003])
def test_fp8_value_dim_64(n, causal):
    """FP8 Q K^T (d = 128) with a 64-wide value head."""
    w = W.Workload("fp8 dv64", 2, 4, n, n, 128, causal, 560 + n, Hkv=2, dv=64)
    q8, k8, v, qd, kd = W.make_qkv_fp8(w)
    assert v.shape[3] == 64
    o, lse = run_fp8(q8, k8, v, causal, w.scale, qd, kd)
    qo, ko, vo = oracle_inputs(q8, k8, v)
    ref = oracle.attention(qo, ko, vo, causal=causal, scale=w.scale * qd * kd)
    compare(o, lse, *ref, f"fp8 dv=64 n={n} causal={causal}")


def test_fp8_query_offset():
    w = W.Workload("fp8 offset", 1, 2, 300, 1000, 128, True, 551)
    q8, k8, v, qd, kd = W.make_qkv_fp8(w)
    o, lse = run_fp8(q8, k8, v, True, w.scale, qd, kd, query_offset=700)
    qo, ko, vo = oracle_inputs(q8, k8, v)
    ref = oracle.attention(qo, ko, vo, causal=True, scale=w.scale * qd * kd, query_offset=700)
    compare(o, lse, *ref, "fp8 offset")


@pytest.mark.parametrize("wl", [W.LONG_PREFILL_CAUSAL, W.LONG_PREFILL_NONCAUSAL],
                         ids=["causal", "noncausal"])
def test_fp8_long_prefill_full_size(wl):
    q8, k8, v, qd, kd = W.make_qkv_fp8(wl)
    o, lse = run_fp8(q8, k8, v, wl.causal, wl.scale, qd, kd)
    rng = np.random.default_rng(3)
    BH = wl.B * wl.H
    heads = sorted({0, BH - 1, *rng.choice(BH, 4, replace=False).tolist()})
    edge = [0, 127, 128, 255, 256, wl.Nq // 2, wl.Nq - 1]
    rows = np.array([h * wl.Nq + i for h in heads
                     for i in sorted(set(edge) | set(rng.integers(0, wl.Nq, 12).tolist()))])
    qo, ko, vo = oracle_inputs(q8, k8, v)
    o_ref, lse_ref = oracle.attention(qo, ko, vo, causal=wl.causal, scale=wl.scale * qd * kd,
                                      rows=rows)
    idx = torch.as_tensor(rows, device=o.device)
    compare(o.reshape(-1, wl.d)[idx], lse.reshape(-1)[idx], o_ref, lse_ref, wl.name + " fp8")
