"""Oracle for the gated delta rule: plain fp64 CPU implementations.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import this package.  The CUDA
product path (``chunked_gated_delta_04_gb300``) never imports it, and the two
share no code; only the seeded input generator serves both.

Two independent evaluations of the same operator (FlashQLA PR #34, Summary and
"Current status"; the operator is fixed as S_t = exp(g_t) S_{t-1}(I - beta_t k_t
k_t^T) + beta_t v_t k_t^T, o_t = scale * S_t q_t):

* ``recurrent_forward`` / ``recurrent_backward``: the token-by-token recurrence
  and its hand-derived reverse-time gradient, in C (``gdr_oracle.c``), threaded
  over (sequence, q/k head) units.
* ``oracle.chunked``: the 64-token chunked WY form in numpy, forward and backward.

``reference()`` maps the C-ABI contract's tensors (layouts, dtypes, varlen) onto
the recurrence and back.  Every function here is pinned by the ``-m "not gpu"``
tests (finite differences, closed forms at beta = 0 and for orthonormal keys, the
exact-overwrite invariant, chunked-vs-recurrent agreement, identity padding,
linearity, varlen = per-sequence runs, and a hand-worked 2x2 example).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdr_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgdr_oracle.so")
_lib = None
_lock = threading.Lock()
CHUNK = 64


def build(force: bool = False) -> str:
    """Compile gdr_oracle.c into a shared library next to it (gcc -O2, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread", "-o", tmp,
                               _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int64)
            i = ctypes.c_int
            lib.gdr_oracle_forward.argtypes = [i, ip, i, i, i, i, ctypes.c_double, dp, dp, dp, dp, dp, dp,
                                               dp, dp, dp, i]
            lib.gdr_oracle_forward.restype = i
            lib.gdr_oracle_backward.argtypes = [i, ip, i, i, i, i, ctypes.c_double, dp, dp, dp, dp, dp, dp,
                                                dp, dp, dp, dp, dp, dp, dp, dp, i]
            lib.gdr_oracle_backward.restype = i
            _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def chunk_offsets(cu_seqlens) -> np.ndarray:
    """chunk_offset[n] = sum_{n' < n} ceil(L_n' / 64); last entry = total chunks."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    lens = np.diff(cu)
    return np.concatenate([[0], np.cumsum((lens + CHUNK - 1) // CHUNK)]).astype(np.int64)


def recurrent_forward(cu_seqlens, Hk, Hv, scale, q, k, v, g, beta, S0=None, nthreads=None,
                      want_chunks=True):
    """Token-by-token forward.  Packed arrays: q,k [T,Hk,DK]; v [T,Hv,DV]; g,beta [T,Hv];
    S0 [N,Hv,DV,DK] (S orientation) or None.  Returns (o, S_T, S_chunks)."""
    lib = _load()
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    q, k, v, g, beta, S0 = map(_f64, (q, k, v, g, beta, S0))
    Ttot, _, DK = q.shape
    DV = v.shape[2]
    o = np.zeros((Ttot, Hv, DV))
    S_T = np.zeros((N, Hv, DV, DK))
    nch = int(chunk_offsets(cu)[-1])
    S_chunks = np.zeros((nch, Hv, DV, DK)) if want_chunks else None
    rc = lib.gdr_oracle_forward(N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), Hk, Hv, DK, DV,
                                float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0),
                                _ptr(o), _ptr(S_T), _ptr(S_chunks), nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"gdr_oracle_forward failed ({rc})")
    return o, S_T, S_chunks


def recurrent_backward(cu_seqlens, Hk, Hv, scale, q, k, v, g, beta, S0, dO, dS_T, nthreads=None):
    """Reverse-time gradient.  Returns (dq, dk, dv, dg, dbeta, dS0); dS0 in S orientation."""
    lib = _load()
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    q, k, v, g, beta, S0, dO, dS_T = map(_f64, (q, k, v, g, beta, S0, dO, dS_T))
    Ttot, _, DK = q.shape
    DV = v.shape[2]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros((Ttot, Hv, DV))
    dg = np.zeros((Ttot, Hv))
    dbeta = np.zeros((Ttot, Hv))
    dS0 = np.zeros((N, Hv, DV, DK))
    rc = lib.gdr_oracle_backward(N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), Hk, Hv, DK, DV,
                                 float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0),
                                 _ptr(dO), _ptr(dS_T), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta),
                                 _ptr(dS0), nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"gdr_oracle_backward failed ({rc})")
    return dq, dk, dv, dg, dbeta, dS0


def _np(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: widen exactly (bf16 -> fp32 -> fp64)
        return x.detach().cpu().float().double().numpy()
    return np.asarray(x, dtype=np.float64)


def reference(inp: dict, layout: str, backward: bool = True, nthreads=None) -> dict:
    """Evaluate the contract's outputs with the recurrence oracle.

    ``inp`` holds the C-ABI tensors (torch or numpy): q,k [B,T,Hk,DK]; v, dO [B,T,Hv,DV];
    g, beta [B,T,Hv]; optional S0 / dS_T ([N,Hv,DK,DV] for layout "KV", [N,Hv,DV,DK] for
    "VK"); optional cu_seqlens (varlen, B == 1); optional scale.  Values are widened to
    fp64 exactly as given (the bf16-rounded inputs the GPU sees).  Returns fp64 numpy
    arrays in the contract's shapes: o, S_T, h_saved ([n_chunks, Hv, DK, DV], "KV"
    orientation whatever ``layout`` is), and with ``backward`` dq, dk, dv, dg, dbeta, dS0.
    """
    q, k, v, g, beta = (_np(inp[n]) for n in ("q", "k", "v", "g", "beta"))
    B, T, Hk, DK = q.shape
    Hv, DV = v.shape[2], v.shape[3]
    cu = inp.get("cu_seqlens")
    if cu is not None:
        cu = np.asarray(_np(cu), dtype=np.int64)
        assert B == 1
    else:
        cu = np.arange(B + 1, dtype=np.int64) * T
    scale = inp.get("scale")
    if scale is None or scale <= 0:
        scale = 1.0 / np.sqrt(DK)

    def to_S(x):  # contract layout -> S orientation [.., DV, DK]
        if x is None:
            return None
        return np.ascontiguousarray(np.swapaxes(x, -1, -2)) if layout == "KV" else np.ascontiguousarray(x)

    def from_S(x):
        return np.ascontiguousarray(np.swapaxes(x, -1, -2)) if layout == "KV" else x

    S0 = to_S(_np(inp.get("S0")))
    pk = lambda a: a.reshape(B * T, *a.shape[2:])
    o, S_T, S_chunks = recurrent_forward(cu, Hk, Hv, scale, pk(q), pk(k), pk(v), pk(g), pk(beta), S0,
                                         nthreads=nthreads)
    out = {
        "o": o.reshape(B, T, Hv, DV),
        "S_T": from_S(S_T),
        "h_saved": np.ascontiguousarray(np.swapaxes(S_chunks, -1, -2)),
    }
    if backward:
        dO = _np(inp["dO"])
        dST = to_S(_np(inp.get("dS_T")))
        dq, dk, dv, dg, dbeta, dS0 = recurrent_backward(cu, Hk, Hv, scale, pk(q), pk(k), pk(v), pk(g),
                                                        pk(beta), S0, pk(dO), dST, nthreads=nthreads)
        out.update(dq=dq.reshape(B, T, Hk, DK), dk=dk.reshape(B, T, Hk, DK), dv=dv.reshape(B, T, Hv, DV),
                   dg=dg.reshape(B, T, Hv), dbeta=dbeta.reshape(B, T, Hv), dS0=from_S(dS0))
    return out
