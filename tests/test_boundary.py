"""The C-ABI boundary without a GPU: the library loads, exports every entry
point that include/attn.h declares, and rejects bad arguments with the
documented status codes before touching CUDA."""
import ctypes
import math
import os
import re
import subprocess

import pytest

from attention_attn_fwd_07_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")

# Fake, never-dereferenced device addresses (validation rejects before use).
A16 = 0x10000
MIS = 0x10008


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def declared_entry_points():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(attn_\w+)\s*\(", text,
                                 flags=re.M)))


def test_header_declares_the_abi():
    names = declared_entry_points()
    assert set(binding.EXPORTED) <= set(names), names
    assert "attn_fwd" in names and "attn_fwd_splitkv" in names and "attn_combine" in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(attn_\w+)$", out, flags=re.M))
    for name in declared_entry_points():
        assert name in exported, f"{name} declared in attn.h but not exported"
        assert hasattr(lib, name)


def call_fwd(lib, q=A16, k=A16, v=A16, o=A16, lse=A16, B=1, H=1, Nq=8, Nk=8, d=64, causal=0,
             scale=0.125):
    return lib.attn_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), binding.ATTN_ERR_INVALID),
    (dict(lse=0), binding.ATTN_ERR_INVALID),
    (dict(B=0), binding.ATTN_ERR_INVALID),
    (dict(H=-1), binding.ATTN_ERR_INVALID),
    (dict(Nq=0), binding.ATTN_ERR_INVALID),
    (dict(Nk=0), binding.ATTN_ERR_INVALID),
    (dict(scale=float("nan")), binding.ATTN_ERR_INVALID),
    (dict(scale=float("inf")), binding.ATTN_ERR_INVALID),
    (dict(scale=0.0), binding.ATTN_ERR_INVALID),
    (dict(scale=-0.5), binding.ATTN_ERR_INVALID),
    (dict(d=32), binding.ATTN_ERR_UNSUPPORTED),
    (dict(d=80), binding.ATTN_ERR_UNSUPPORTED),
    (dict(d=192), binding.ATTN_ERR_UNSUPPORTED),
    (dict(d=512), binding.ATTN_ERR_UNSUPPORTED),
    (dict(Nq=1 << 31), binding.ATTN_ERR_UNSUPPORTED),
    (dict(B=1 << 20, H=1 << 12), binding.ATTN_ERR_UNSUPPORTED),
    (dict(q=MIS), binding.ATTN_ERR_ALIGN),
    (dict(o=MIS + 4), binding.ATTN_ERR_ALIGN),
    (dict(lse=A16 + 2), binding.ATTN_ERR_ALIGN),
])
def test_fwd_rejects(lib, kw, code):
    assert call_fwd(lib, **kw) == code


def _params(**kw):
    base = dict(q=A16, k=A16, v=A16, o=A16, lse=A16, B=1, H=1, Nq=8, Nk=8, d=64, causal=1,
                scale=0.125, query_offset=0, dev_status=None, flags=0, wait_timeout_us=0, Hkv=0,
                qk_dtype=0, q_descale=0.0, k_descale=0.0, dv=0)
    base.update(kw)
    return binding.attn_params(**base)


def test_negative_offset_needs_flag(lib):
    p = _params(query_offset=-3)
    assert lib.attn_fwd_ex(ctypes.byref(p), None) == binding.ATTN_ERR_INVALID
    p = _params(query_offset=1 << 41, flags=binding.ATTN_FLAG_ALLOW_NEG_OFFSET)
    assert lib.attn_fwd_ex(ctypes.byref(p), None) == binding.ATTN_ERR_INVALID
    assert lib.attn_fwd_ex(None, None) == binding.ATTN_ERR_INVALID


@pytest.mark.parametrize("H,Hkv", [(8, 3), (8, 16), (8, -1), (6, 4)])
def test_grouped_heads_must_divide(lib, H, Hkv):
    p = _params(H=H, Hkv=Hkv)
    assert lib.attn_fwd_ex(ctypes.byref(p), None) == binding.ATTN_ERR_INVALID
    need = lib.attn_splitkv_workspace_bytes(1, H, 8, 64, 2)
    assert lib.attn_fwd_splitkv_ex(ctypes.byref(p), 2, A16, need, None) == binding.ATTN_ERR_INVALID


@pytest.mark.parametrize("kw,code", [
    (dict(qk_dtype=1, q_descale=1.0, k_descale=1.0, d=64), binding.ATTN_ERR_UNSUPPORTED),
    (dict(qk_dtype=1, q_descale=1.0, k_descale=1.0, d=96), binding.ATTN_ERR_UNSUPPORTED),
    (dict(qk_dtype=1, q_descale=1.0, k_descale=1.0, d=256), binding.ATTN_ERR_UNSUPPORTED),
    (dict(qk_dtype=1, q_descale=0.0, k_descale=1.0, d=128), binding.ATTN_ERR_INVALID),
    (dict(qk_dtype=1, q_descale=1.0, k_descale=float("nan"), d=128), binding.ATTN_ERR_INVALID),
    (dict(qk_dtype=2, q_descale=1.0, k_descale=1.0, d=128), binding.ATTN_ERR_INVALID),
])
def test_fp8_arguments(lib, kw, code):
    p = _params(**kw)
    assert lib.attn_fwd_ex(ctypes.byref(p), None) == code
    if code == binding.ATTN_ERR_UNSUPPORTED:
        need = lib.attn_splitkv_workspace_bytes(1, 1, 8, 64, 2)
        assert lib.attn_fwd_splitkv_ex(ctypes.byref(p), 2, A16, need, None) == code


def test_workspace_bytes(lib):
    f = lib.attn_splitkv_workspace_bytes
    rows = 16 * 32 * 64 * 1
    assert f(16, 32, 1, 128, 64) == math.ceil(rows * 128 * 4 / 256) * 256 + rows * 4
    rows = 3 * 4 * 3 * 1003
    assert f(3, 4, 1003, 64, 3) == math.ceil(rows * 64 * 4 / 256) * 256 + rows * 4
    for d in (96, 256):  # every head dim the forward takes has a workspace size
        assert f(2, 3, 5, d, 7) == math.ceil(2 * 3 * 7 * 5 * d * 4 / 256) * 256 + 2 * 3 * 7 * 5 * 4
    for bad in [(0, 1, 1, 64, 1), (1, 1, 1, 80, 1), (1, 1, 1, 32, 1), (1, 1, 1, 64, 0),
                (1, 1, 1, 64, 257), (1, 1, 0, 64, 1)]:
        assert f(*bad) == 0


def test_splitkv_rejects(lib):
    need = lib.attn_splitkv_workspace_bytes(1, 1, 8, 64, 4)
    sk = lib.attn_fwd_splitkv
    args = [A16, A16, A16, A16, A16, 1, 1, 8, 8, 64, 0, 0.125]
    assert sk(*args, 0, A16, need, None) == binding.ATTN_ERR_INVALID
    assert sk(*args, 257, A16, need, None) == binding.ATTN_ERR_INVALID
    assert sk(*args, 4, 0, need, None) == binding.ATTN_ERR_WORKSPACE
    assert sk(*args, 4, A16, need - 1, None) == binding.ATTN_ERR_WORKSPACE
    assert sk(*args, 4, MIS, need, None) == binding.ATTN_ERR_ALIGN
    bad = list(args)
    bad[9] = 80
    assert sk(*bad, 4, A16, need, None) == binding.ATTN_ERR_UNSUPPORTED


def test_noalloc_rejects(lib):
    """The allocation-free split-KV entry point shares the workspace entry
    point's checks, refuses the head dims its CUDA-core kernels do not cover
    and problems whose scratch exceeds its fixed array -- all before any CUDA
    call."""
    f = lib.attn_fwd_splitkv_noalloc
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64] * 5 + [ctypes.c_int, ctypes.c_float,
                                                                 ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    args = [A16, A16, A16, A16, A16, 1, 1, 8, 8]
    assert f(*args, 64, 0, 0.125, 0, None) == binding.ATTN_ERR_INVALID
    assert f(*args, 64, 0, float("nan"), 4, None) == binding.ATTN_ERR_INVALID
    assert f(MIS, *args[1:], 64, 0, 0.125, 4, None) == binding.ATTN_ERR_ALIGN
    for d in (96, 256):
        assert f(*args, d, 0, 0.125, 4, None) == binding.ATTN_ERR_UNSUPPORTED
    assert f(*args, 80, 0, 0.125, 4, None) == binding.ATTN_ERR_UNSUPPORTED
    big = [A16, A16, A16, A16, A16, 16, 32, 1, 4096]
    assert f(*big, 128, 0, 0.125, 128, None) == binding.ATTN_ERR_WORKSPACE


def test_from_host_rejects(lib):
    """The host-buffer entry point applies the forward's checks and its own
    (host pointers, chunk size, FP8) before any CUDA call."""
    f = lib.attn_fwd_from_host
    host = ctypes.create_string_buffer(64)
    hp = ctypes.addressof(host)
    p = _params()
    assert f(ctypes.byref(p), hp, hp, hp, hp, hp, 0, None, None, None) == binding.ATTN_ERR_INVALID
    assert f(ctypes.byref(p), 0, hp, hp, hp, hp, 8, None, None, None) == binding.ATTN_ERR_INVALID
    assert f(ctypes.byref(p), hp, hp, hp, hp, 0, 8, None, None, None) == binding.ATTN_ERR_INVALID
    bad = _params(d=80)
    assert f(ctypes.byref(bad), hp, hp, hp, hp, hp, 8, None, None, None) == \
        binding.ATTN_ERR_UNSUPPORTED
    fp8 = _params(d=128, qk_dtype=1, q_descale=1.0, k_descale=1.0)
    assert f(ctypes.byref(fp8), hp, hp, hp, hp, hp, 8, None, None, None) == \
        binding.ATTN_ERR_UNSUPPORTED
    mis = _params(q=MIS)
    assert f(ctypes.byref(mis), hp, hp, hp, hp, hp, 8, None, None, None) == binding.ATTN_ERR_ALIGN
    assert f(None, hp, hp, hp, hp, hp, 8, None, None, None) == binding.ATTN_ERR_INVALID


def test_combine_rejects(lib):
    c = lib.attn_combine
    assert c(0, A16, A16, A16, 1, 1, 1, 64, 4, None) == binding.ATTN_ERR_INVALID
    assert c(A16, A16, A16, A16, 1, 1, 1, 64, 0, None) == binding.ATTN_ERR_INVALID
    assert c(A16, A16, A16, A16, 1, 1, 1, 32, 4, None) == binding.ATTN_ERR_UNSUPPORTED
    assert c(A16, A16, A16, A16, 1, 1, 1, 80, 4, None) == binding.ATTN_ERR_UNSUPPORTED
    assert c(MIS, A16, A16, A16, 1, 1, 1, 64, 4, None) == binding.ATTN_ERR_ALIGN


def test_status_strings(lib):
    for code in range(-6, 1):
        s = lib.attn_status_string(code).decode()
        assert s.startswith("ATTN_")
    assert "unknown" in lib.attn_status_string(42).decode()
    assert lib.attn_get_device_status(None, None) == binding.ATTN_ERR_INVALID


def test_valid_call_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("only meaningful on a host without a GPU (fake pointers)")
    assert call_fwd(lib) == binding.ATTN_ERR_CUDA


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        binding.load_library(str(tmp_path / "nope.so"))


def _bwd_params(**kw):
    base = dict(q=A16, k=A16, v=A16, o=A16, dout=A16, lse=A16, dq=A16, dk=A16, dv=A16, B=1, H=2,
                Hkv=0, Nq=8, Nk=8, d=128, causal=1, scale=0.125, query_offset=0,
                dev_status=None, flags=0, wait_timeout_us=0, value_dim=0)
    base.update(kw)
    return binding.attn_bwd_params(**base)


@pytest.mark.parametrize("kw,ws,code", [
    (dict(q=0), 1 << 20, binding.ATTN_ERR_INVALID),
    (dict(dout=0), 1 << 20, binding.ATTN_ERR_INVALID),
    (dict(dk=0), 1 << 20, binding.ATTN_ERR_INVALID),
    (dict(Nq=0), 1 << 20, binding.ATTN_ERR_INVALID),
    (dict(scale=float("nan")), 1 << 20, binding.ATTN_ERR_INVALID),
    (dict(Hkv=3), 1 << 20, binding.ATTN_ERR_INVALID),
    (dict(Hkv=4), 1 << 20, binding.ATTN_ERR_INVALID),
    (dict(query_offset=-1), 1 << 20, binding.ATTN_ERR_INVALID),
    (dict(d=96, value_dim=64), 1 << 20, binding.ATTN_ERR_UNSUPPORTED),
    (dict(d=96, value_dim=128), 1 << 20, binding.ATTN_ERR_UNSUPPORTED),
    (dict(d=256), 1 << 20, binding.ATTN_ERR_UNSUPPORTED),
    (dict(value_dim=-1), 1 << 20, binding.ATTN_ERR_INVALID),
    (dict(value_dim=96), 1 << 20, binding.ATTN_ERR_UNSUPPORTED),
    (dict(value_dim=256), 1 << 20, binding.ATTN_ERR_UNSUPPORTED),
    (dict(Nq=1 << 31), 1 << 20, binding.ATTN_ERR_UNSUPPORTED),
    (dict(dq=MIS), 1 << 20, binding.ATTN_ERR_ALIGN),
    (dict(lse=A16 + 2), 1 << 20, binding.ATTN_ERR_ALIGN),
    (dict(), 16, binding.ATTN_ERR_WORKSPACE),
])
def test_bwd_rejects(lib, kw, ws, code):
    p = _bwd_params(**kw)
    assert lib.attn_bwd(ctypes.byref(p), A16, ws, None) == code


def test_bwd_workspace_bytes(lib):
    assert lib.attn_bwd_workspace_bytes(2, 3, 100) >= 2 * 3 * 100 * 4
    assert lib.attn_bwd_workspace_bytes(2, 3, 100) % 256 == 0
    assert lib.attn_bwd_workspace_bytes(0, 3, 100) == 0
    assert lib.attn_bwd(None, A16, 1 << 20, None) == binding.ATTN_ERR_INVALID


@pytest.mark.parametrize("kw,code", [
    (dict(dv=-1), binding.ATTN_ERR_INVALID),
    (dict(dv=96), binding.ATTN_ERR_UNSUPPORTED),
    (dict(dv=256), binding.ATTN_ERR_UNSUPPORTED),
    (dict(d=96, dv=64), binding.ATTN_ERR_UNSUPPORTED),
    (dict(d=256, dv=128), binding.ATTN_ERR_UNSUPPORTED),
    (dict(d=128, dv=96), binding.ATTN_ERR_UNSUPPORTED),
    (dict(d=64, dv=128, qk_dtype=1, q_descale=1.0, k_descale=1.0), binding.ATTN_ERR_UNSUPPORTED),
])
def test_value_dim_rejects(lib, kw, code):
    p = _params(**kw)
    assert lib.attn_fwd_ex(ctypes.byref(p), None) == code


def test_splitkv_value_dim_workspace(lib):
    # Split-KV partials are as wide as V: a workspace sized for d is too
    # small when dv > d, and value dims other than 64 and 128 are refused.
    small = lib.attn_splitkv_workspace_bytes(1, 1, 8, 64, 4)
    need = lib.attn_splitkv_workspace_bytes(1, 1, 8, 128, 4)
    assert need > small > 0
    p = _params(d=64, dv=128)
    assert lib.attn_fwd_splitkv_ex(ctypes.byref(p), 4, A16, small, None) == \
        binding.ATTN_ERR_WORKSPACE
    p = _params(d=64, dv=96)
    assert lib.attn_fwd_splitkv_ex(ctypes.byref(p), 4, A16, 1 << 30, None) == \
        binding.ATTN_ERR_UNSUPPORTED
