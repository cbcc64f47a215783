"""TEST INFRASTRUCTURE ONLY: the CPU fp64 attention oracle.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  It shares no code with the CUDA
library and never imports it.

``attention`` is the dense definition of softmax attention from
"GPU Engineering: Correctness, Throughput, and Attention" (section 22.7, the
worked tiled-attention lab: causal rule ``j > i + query_offset``, rows with no
admissible key give output 0 and log-normaliser -inf; section 22.5: tiling
with rescaling reaches the full stable softmax in real arithmetic), computed
in IEEE double by ``oracle.c``.

Pins that tie it to the pages and to mathematics live in
``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SRC_BWD = os.path.join(_HERE, "oracle_bwd.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F64, BF16 = 0, 1


def build(out_path: str = _LIB_PATH, plant: int = 0) -> str:
    """Compile oracle.c with gcc (IEEE semantics: no fast-math, no -march).

    ``plant`` > 0 builds a deliberately wrong variant for the pin tests.
    """
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", _SRC, _SRC_BWD, "-o", out_path, "-lm"]
    if plant:
        cmd.insert(1, f"-DORACLE_PLANT={int(plant)}")
    subprocess.run(cmd, check=True)
    return out_path


def _stale() -> bool:
    return (not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                                 os.path.getmtime(_SRC_BWD)))


def load(path: str | None = None):
    """Load (building if needed) the oracle shared library."""
    global _lib
    if path is not None:
        lib = ctypes.CDLL(path)
        _declare(lib)
        return lib
    with _lock:
        if _lib is None:
            if _stale():
                build()
            _lib = ctypes.CDLL(_LIB_PATH)
            _declare(_lib)
    return _lib


def _declare(lib) -> None:
    f = lib.oracle_attention
    f.restype = ctypes.c_int
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    f.argtypes = [vp, vp, vp, ctypes.c_int, i64, i64, i64, i64, i64, i64, i64,
                  ctypes.c_int, i64, ctypes.c_double, i64, i64, vp, i64, vp,
                  vp, ctypes.c_int]
    lib.oracle_plant.restype = ctypes.c_int
    b = lib.oracle_attention_bwd
    b.restype = ctypes.c_int
    b.argtypes = [vp, vp, vp, vp, ctypes.c_int, i64, i64, i64, i64, i64, i64, i64, ctypes.c_int,
                  i64, ctypes.c_double, vp, vp, vp, ctypes.c_int]


def _as_array(x):
    """Return (contiguous numpy array, element code) for f64 or bf16 input.

    bf16 may be given as a torch.bfloat16 CPU tensor or as uint16 bit
    patterns; anything else floating is converted to float64.
    """
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return np.ascontiguousarray(x.view(torch.int16).numpy().view(np.uint16)), BF16
            return np.ascontiguousarray(x.to(torch.float64).numpy()), F64
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return np.ascontiguousarray(x), BF16
    return np.ascontiguousarray(x, dtype=np.float64), F64


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def attention(q, k, v, *, causal: bool, scale: float, query_offset: int = 0,
              key_range: tuple[int, int] | None = None, rows=None,
              threads: int | None = None, lib=None):
    """Dense fp64 softmax attention over 4-D [B, H, N, dim] inputs.

    K and V may have fewer heads than Q (grouped K/V heads): query head h
    reads K/V head h // (H // Hkv).

    Returns ``(o, lse)`` as float64 numpy arrays.  With ``rows`` = None, o has
    shape [B, H, Nq, dv] and lse [B, H, Nq]; with ``rows`` (flattened indices
    (b*H + h)*Nq + i) they have shapes [len(rows), dv] and [len(rows)].
    ``scale`` is used as given (callers pass the fp32 value the GPU sees).
    """
    lib = lib or load()
    qa, qe = _as_array(q)
    ka, ke = _as_array(k)
    va, ve = _as_array(v)
    if not (qe == ke == ve):
        raise ValueError("q, k and v must share one element type")
    if qa.ndim != 4 or ka.ndim != 4 or va.ndim != 4:
        raise ValueError("expected [B, H, N, dim] inputs")
    B, H, Nq, d = qa.shape
    Bk, Hkv, Nk, dk = ka.shape
    if (Bk, dk) != (B, d) or va.shape[:3] != (B, Hkv, Nk) or Hkv < 1 or H % Hkv != 0:
        raise ValueError("incompatible q, k, v shapes")
    dv = va.shape[3]
    lo, hi = key_range if key_range is not None else (0, Nk)
    if rows is not None:
        rows_a = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).ravel())
        n_out = rows_a.size
        rows_p = rows_a.ctypes.data
    else:
        rows_a = None
        n_out = B * H * Nq
        rows_p = None
    o = np.empty((n_out, dv), dtype=np.float64)
    lse = np.empty((n_out,), dtype=np.float64)
    rc = lib.oracle_attention(
        qa.ctypes.data, ka.ctypes.data, va.ctypes.data, qe, B, H, Hkv, Nq, Nk, d, dv,
        int(bool(causal)), int(query_offset), float(scale), int(lo), int(hi),
        rows_p, n_out if rows_a is not None else 0, o.ctypes.data,
        lse.ctypes.data, int(threads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_attention rejected its arguments (status {rc})")
    if rows_a is None:
        return o.reshape(B, H, Nq, dv), lse.reshape(B, H, Nq)
    return o, lse


def attention_bwd(q, k, v, dout, *, causal: bool, scale: float, query_offset: int = 0,
                  threads: int | None = None, lib=None):
    """Dense fp64 gradients (dq, dk, dv) of softmax attention for the loss
    gradient ``dout`` on O; q [B, H, Nq, d], k [B, Hkv, Nk, d], v
    [B, Hkv, Nk, dv], dout [B, H, Nq, dv] (dv may differ from d)."""
    lib = lib or load()
    qa, qe = _as_array(q)
    ka, ke = _as_array(k)
    va, ve = _as_array(v)
    da, de = _as_array(dout)
    if not (qe == ke == ve == de):
        raise ValueError("q, k, v and dout must share one element type")
    B, H, Nq, d = qa.shape
    Bk, Hkv, Nk, dk_ = ka.shape
    e = va.shape[3]
    if ((Bk, dk_) != (B, d) or va.shape[:3] != ka.shape[:3] or da.shape != (B, H, Nq, e)
            or H % Hkv != 0):
        raise ValueError("incompatible shapes")
    dq = np.empty((B, H, Nq, d), dtype=np.float64)
    dk = np.empty((B, Hkv, Nk, d), dtype=np.float64)
    dv = np.empty((B, Hkv, Nk, e), dtype=np.float64)
    rc = lib.oracle_attention_bwd(qa.ctypes.data, ka.ctypes.data, va.ctypes.data,
                                  da.ctypes.data, qe, B, H, Hkv, Nq, Nk, d, e, int(bool(causal)),
                                  int(query_offset), float(scale), dq.ctypes.data,
                                  dk.ctypes.data, dv.ctypes.data,
                                  int(threads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_attention_bwd rejected its arguments (status {rc})")
    return dq, dk, dv
