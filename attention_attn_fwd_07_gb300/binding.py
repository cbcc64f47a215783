"""ctypes binding of the C ABI in ``include/attn.h``.

Argument marshalling only: every function here checks Python-side types,
takes raw device pointers from torch tensors, and calls the C entry point of
the same name on the caller's current CUDA stream.  All computation runs in
the library's kernels.  If ``libattn_gb300.so`` is missing the first call
raises; there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn_gb300.so")
_lock = threading.Lock()
_lib = None

ATTN_OK = 0
ATTN_ERR_INVALID = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_ALIGN = -3
ATTN_ERR_WORKSPACE = -4
ATTN_ERR_CUDA = -5
ATTN_ERR_DEVICE_TIMEOUT = -6
ATTN_FLAG_ALLOW_NEG_OFFSET = 1 << 0
ATTN_FLAG_TEST_SKIP_LOAD = 1 << 1
ATTN_QK_BF16 = 0
ATTN_QK_E4M3 = 1

EXPORTED = ("attn_fwd", "attn_fwd_ex", "attn_fwd_splitkv", "attn_fwd_splitkv_ex",
            "attn_combine", "attn_splitkv_workspace_bytes", "attn_get_device_status",
            "attn_status_string", "attn_bwd", "attn_bwd_workspace_bytes",
            "attn_fwd_from_host")


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {attn_status_string(status)} ({status})")


class attn_params(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("B", ctypes.c_int64), ("H", ctypes.c_int64), ("Nq", ctypes.c_int64),
                ("Nk", ctypes.c_int64), ("d", ctypes.c_int64),
                ("causal", ctypes.c_int), ("scale", ctypes.c_float),
                ("query_offset", ctypes.c_int64), ("dev_status", ctypes.c_void_p),
                ("flags", ctypes.c_uint32), ("wait_timeout_us", ctypes.c_uint32),
                ("Hkv", ctypes.c_int64), ("qk_dtype", ctypes.c_int),
                ("q_descale", ctypes.c_float), ("k_descale", ctypes.c_float),
                ("dv", ctypes.c_int64)]


class attn_bwd_params(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("o", ctypes.c_void_p), ("dout", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
                ("B", ctypes.c_int64), ("H", ctypes.c_int64), ("Hkv", ctypes.c_int64),
                ("Nq", ctypes.c_int64), ("Nk", ctypes.c_int64), ("d", ctypes.c_int64),
                ("causal", ctypes.c_int), ("scale", ctypes.c_float),
                ("query_offset", ctypes.c_int64), ("dev_status", ctypes.c_void_p),
                ("flags", ctypes.c_uint32), ("wait_timeout_us", ctypes.c_uint32),
                ("value_dim", ctypes.c_int64)]


def load_library(path: str | None = None):
    """Load the CUDA library (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build it with `python -m attention_attn_fwd_07_gb300.build`")
        lib = ctypes.CDLL(p)
        i64, vp, c_int, c_float = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, c_int, c_float, vp]
        lib.attn_fwd.restype = c_int
        lib.attn_fwd_ex.argtypes = [ctypes.POINTER(attn_params), vp]
        lib.attn_fwd_ex.restype = c_int
        lib.attn_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, c_int,
                                         c_float, c_int, vp, ctypes.c_size_t, vp]
        lib.attn_fwd_splitkv.restype = c_int
        lib.attn_fwd_splitkv_ex.argtypes = [ctypes.POINTER(attn_params), c_int, vp,
                                            ctypes.c_size_t, vp]
        lib.attn_fwd_splitkv_ex.restype = c_int
        lib.attn_splitkv_workspace_bytes.argtypes = [i64, i64, i64, i64, c_int]
        lib.attn_splitkv_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_combine.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, c_int, vp]
        lib.attn_combine.restype = c_int
        lib.attn_get_device_status.argtypes = [ctypes.POINTER(c_int), vp]
        lib.attn_get_device_status.restype = c_int
        lib.attn_bwd.argtypes = [ctypes.POINTER(attn_bwd_params), vp, ctypes.c_size_t, vp]
        lib.attn_bwd.restype = c_int
        lib.attn_bwd_workspace_bytes.argtypes = [i64, i64, i64]
        lib.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_fwd_from_host.argtypes = [ctypes.POINTER(attn_params), vp, vp, vp, vp, vp,
                                           c_int, vp, vp, vp]
        lib.attn_fwd_from_host.restype = c_int
        lib.attn_status_string.argtypes = [c_int]
        lib.attn_status_string.restype = ctypes.c_char_p
        if path is None:
            _lib = lib
        return lib


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, torch.Tensor):
        return t.data_ptr()
    return int(t)


def _check(rc: int, what: str) -> None:
    if rc != ATTN_OK:
        raise AttnError(rc, what)


def _require(t, dtype, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _shape(q, k, v=None):
    """(B, H, Nq, Nk, d) of q [B, H, Nq, d], k [B, Hkv, Nk, d], v [B, Hkv, Nk, dv]."""
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    _require(q, torch.bfloat16, "q")
    _require(k, torch.bfloat16, "k")
    if v is not None:
        _require(v, torch.bfloat16, "v")
        if v.dim() != 4 or tuple(v.shape[:3]) != tuple(k.shape[:3]):
            raise ValueError("v must be [B, Hkv, Nk, dv] with the batch, heads and keys of k")
    B, H, Nq, d = q.shape
    if k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k must be [B, Hkv, Nk, d] with the batch and head dim of q")
    return B, H, Nq, k.shape[2], d


def _outputs(q, o, lse, dv=None):
    B, H, Nq, d = q.shape
    if o is None:
        o = torch.empty((B, H, Nq, dv or d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    _require(o, torch.bfloat16, "o")
    _require(lse, torch.float32, "lse")
    return o, lse


def attn_fwd(q, k, v, causal: bool, scale: float, o=None, lse=None, stream=None):
    """Prefill forward: returns (o bf16 [B,H,Nq,d], lse f32 [B,H,Nq]).

    K/V with fewer heads than Q (grouped K/V heads) go through attn_fwd_ex."""
    B, H, Nq, Nk, d = _shape(q, k, v)
    if k.shape[1] != H or v.shape[3] != d:
        return attn_fwd_ex(q, k, v, causal, scale, o=o, lse=lse, stream=stream)
    o, lse = _outputs(q, o, lse)
    rc = load_library().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d,
                                 int(bool(causal)), float(scale), _stream(stream))
    _check(rc, "attn_fwd")
    return o, lse


def make_params(q, k, v, o, lse, causal, scale, query_offset=0, flags=0, dev_status=None,
                wait_timeout_us=0) -> attn_params:
    B, H, Nq, Nk, d = _shape(q, k, v)
    return attn_params(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d,
                       int(bool(causal)), float(scale), int(query_offset), _ptr(dev_status),
                       int(flags), int(wait_timeout_us), int(k.shape[1]), dv=int(v.shape[3]))


def attn_fwd_ex(q, k, v, causal: bool, scale: float, query_offset: int = 0, flags: int = 0,
                dev_status=None, wait_timeout_us: int = 0, o=None, lse=None, stream=None):
    o, lse = _outputs(q, o, lse, dv=v.shape[3])
    p = make_params(q, k, v, o, lse, causal, scale, query_offset, flags, dev_status,
                    wait_timeout_us)
    _check(load_library().attn_fwd_ex(ctypes.byref(p), _stream(stream)), "attn_fwd_ex")
    return o, lse


def attn_fwd_fp8(q8, k8, v, causal: bool, scale: float, q_descale: float, k_descale: float,
                 query_offset: int = 0, o=None, lse=None, stream=None):
    """Prefill with FP8 Q K^T: q8 [B,H,Nq,128], k8 [B,Hkv,Nk,128] e4m3 codes
    (uint8 or float8_e4m3fn tensors), v bf16 [B,Hkv,Nk,dv] (dv 64 or 128);
    scores are scale * q_descale * k_descale * <q, k>.  Calls attn_fwd_ex."""
    for name, t in (("q8", q8), ("k8", k8)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
        if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
            raise ValueError(f"{name} must hold e4m3 codes (uint8 or float8_e4m3fn)")
    _require(v, torch.bfloat16, "v")
    B, H, Nq, d = q8.shape
    if (k8.dim() != 4 or v.dim() != 4 or tuple(v.shape[:3]) != tuple(k8.shape[:3])
            or k8.shape[0] != B or k8.shape[3] != d):
        raise ValueError("k8 must be [B, Hkv, Nk, d] and v [B, Hkv, Nk, dv]")
    dv = v.shape[3]
    if o is None:
        o = torch.empty((B, H, Nq, dv), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q8.device)
    _require(o, torch.bfloat16, "o")
    _require(lse, torch.float32, "lse")
    p = attn_params(_ptr(q8), _ptr(k8), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, k8.shape[2], d,
                    int(bool(causal)), float(scale), int(query_offset), 0, 0, 0,
                    int(k8.shape[1]), ATTN_QK_E4M3, float(q_descale), float(k_descale), int(dv))
    _check(load_library().attn_fwd_ex(ctypes.byref(p), _stream(stream)), "attn_fwd_ex (fp8)")
    return o, lse


def attn_splitkv_workspace_bytes(B: int, H: int, Nq: int, d: int, num_splits: int) -> int:
    return int(load_library().attn_splitkv_workspace_bytes(B, H, Nq, d, num_splits))


def _workspace(q, num_splits, workspace, dv=None):
    """Split-KV workspace (partials are as wide as V: ``dv``, default d)."""
    B, H, Nq, d = q.shape
    need = attn_splitkv_workspace_bytes(B, H, Nq, dv or d, num_splits)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=q.device)
    return workspace, workspace.numel() * workspace.element_size()


def attn_fwd_splitkv(q, k, v, causal: bool, scale: float, num_splits: int, workspace=None,
                     o=None, lse=None, stream=None):
    """Split-KV forward (partial + combine).  ``workspace``: caller's uint8 tensor.

    K/V with fewer heads than Q (grouped K/V heads) go through attn_fwd_splitkv_ex."""
    B, H, Nq, Nk, d = _shape(q, k, v)
    if k.shape[1] != H or v.shape[3] != d:
        return attn_fwd_splitkv_ex(q, k, v, causal, scale, num_splits, workspace=workspace,
                                   o=o, lse=lse, stream=stream)
    o, lse = _outputs(q, o, lse)
    ws, ws_bytes = _workspace(q, num_splits, workspace)
    rc = load_library().attn_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq,
                                         Nk, d, int(bool(causal)), float(scale), int(num_splits),
                                         _ptr(ws), ws_bytes, _stream(stream))
    _check(rc, "attn_fwd_splitkv")
    return o, lse


def attn_fwd_splitkv_ex(q, k, v, causal: bool, scale: float, num_splits: int,
                        query_offset: int = 0, flags: int = 0, workspace=None, o=None, lse=None,
                        stream=None):
    dv = v.shape[3]
    o, lse = _outputs(q, o, lse, dv)
    ws, ws_bytes = _workspace(q, num_splits, workspace, dv)
    p = make_params(q, k, v, o, lse, causal, scale, query_offset, flags)
    rc = load_library().attn_fwd_splitkv_ex(ctypes.byref(p), int(num_splits), _ptr(ws), ws_bytes,
                                            _stream(stream))
    _check(rc, "attn_fwd_splitkv_ex")
    return o, lse


def attn_combine(o_part, lse_part, num_splits: int, o=None, lse=None, stream=None):
    """Merge partial states: o_part f32 [B,H,S,Nq,d], lse_part f32 [B,H,S,Nq]."""
    _require(o_part, torch.float32, "o_part")
    _require(lse_part, torch.float32, "lse_part")
    B, H, S, Nq, d = o_part.shape
    if S != num_splits or tuple(lse_part.shape) != (B, H, S, Nq):
        raise ValueError("o_part / lse_part shapes do not match num_splits")
    if o is None:
        o = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=o_part.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=o_part.device)
    rc = load_library().attn_combine(_ptr(o_part), _ptr(lse_part), _ptr(o), _ptr(lse), B, H, Nq,
                                     d, int(num_splits), _stream(stream))
    _check(rc, "attn_combine")
    return o, lse


def attn_get_device_status(stream=None) -> int:
    """Synchronise, read and clear the library's device status word."""
    out = ctypes.c_int(0)
    _check(load_library().attn_get_device_status(ctypes.byref(out), _stream(stream)),
           "attn_get_device_status")
    return out.value


_side_streams: dict = {}


def _streams_for(device):
    """Two side streams per device (uploads, downloads), created once."""
    key = torch.device(device).index
    if key not in _side_streams:
        _side_streams[key] = (torch.cuda.Stream(device=device), torch.cuda.Stream(device=device))
    return _side_streams[key]


def fwd_from_host(q_host, k_host, v_host, causal: bool, scale: float, q_dev, k_dev, v_dev,
                  o_dev, lse_dev, o_host, lse_host, stream=None, chunk_heads: int = 8):
    """End-to-end call with pinned host buffers (the C entry point
    attn_fwd_from_host): host -> device copies of Q, K, V, the forward,
    device -> host copies of O and LSE, pipelined in chunks of
    ``chunk_heads`` query heads of one batch entry over an upload stream,
    ``stream`` and a download stream (two side streams per device, created
    once here).  ``stream`` waits for the last download before this returns
    (the host buffers are valid once ``stream`` is synchronised)."""
    for t, name in ((q_host, "q_host"), (k_host, "k_host"), (v_host, "v_host"),
                    (o_host, "o_host"), (lse_host, "lse_host")):
        if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor")
    if (q_host.shape != q_dev.shape or k_host.shape != k_dev.shape or v_host.shape != v_dev.shape
            or o_host.shape != o_dev.shape or lse_host.shape != lse_dev.shape):
        raise ValueError("host and device tensors must have the same shapes")
    up, down = _streams_for(q_dev.device)
    p = make_params(q_dev, k_dev, v_dev, o_dev, lse_dev, causal, scale)
    rc = load_library().attn_fwd_from_host(
        ctypes.byref(p), _ptr(q_host), _ptr(k_host), _ptr(v_host), _ptr(o_host), _ptr(lse_host),
        int(chunk_heads), _stream(stream), up.cuda_stream, down.cuda_stream)
    _check(rc, "attn_fwd_from_host")
    return o_host, lse_host


def attn_bwd_workspace_bytes(B: int, H: int, Nq: int) -> int:
    return int(load_library().attn_bwd_workspace_bytes(B, H, Nq))


def attn_bwd(q, k, v, o, lse, dout, causal: bool, scale: float, query_offset: int = 0,
             flags: int = 0, workspace=None, dq=None, dk=None, dv=None, stream=None):
    """Backward pass: returns (dq, dk, dv) bf16 for the loss gradient dout on o."""
    B, H, Nq, Nk, d = _shape(q, k, v)
    dvw = v.shape[3]  # value head dim: V, O, dO and dV
    _require(o, torch.bfloat16, "o")
    _require(dout, torch.bfloat16, "dout")
    _require(lse, torch.float32, "lse")
    if tuple(o.shape) != (B, H, Nq, dvw) or tuple(dout.shape) != (B, H, Nq, dvw):
        raise ValueError("o and dout must be [B, H, Nq, dv]")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _require(t, torch.bfloat16, name)
    need = attn_bwd_workspace_bytes(B, H, Nq)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=q.device)
    p = attn_bwd_params(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                        _ptr(dk), _ptr(dv), B, H, k.shape[1], Nq, Nk, d, int(bool(causal)),
                        float(scale), int(query_offset), 0, int(flags), 0, int(dvw))
    rc = load_library().attn_bwd(ctypes.byref(p), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "attn_bwd")
    return dq, dk, dv
