"""chunked_gated_delta_04_gb300 -- the chunked gated delta rule on GB300 (sm_103a).

A thin ctypes binding over ``libgdr.so`` (C ABI in ``include/gdr.h``).  The entry
points keep the C names (``gdr_fwd``, ``gdr_bwd``, ...) and only marshal
arguments: every step of the computation runs in the library's CUDA kernels.
PyTorch supplies device memory and the current stream.  There is no CPU path:
if the library cannot be loaded, every call raises.

Operator (FlashQLA PR #34, "SM120/121: Add support for fused backward kernel",
Summary and "Current status"): S_t = exp(g_t) S_{t-1}(I - beta_t k_t k_t^T) +
beta_t v_t k_t^T, o_t = scale * S_t q_t, evaluated in 64-token chunks, with its
backward (dq, dk, dv, dg, dbeta, dS0 from dO and dS_T).

High-level helpers: ``forward`` / ``backward`` allocate outputs and workspace with
torch; ``chunk_gated_delta_rule`` is the autograd entry point.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdr.so")

GDR_OK, GDR_ERR_INVALID_ARG, GDR_ERR_UNSUPPORTED, GDR_ERR_ALIGNMENT, GDR_ERR_CUDA, GDR_ERR_TIMEOUT, \
    GDR_ERR_WORKSPACE = range(7)
GDR_DTYPE_F32, GDR_DTYPE_BF16 = 0, 1
GDR_STATE_KV, GDR_STATE_VK = 0, 1
GDR_PROLOGUE_QK_L2NORM, GDR_PROLOGUE_G_LOGSIGMOID, GDR_PROLOGUE_BETA_SIGMOID = 1, 2, 4
GDR_PROLOGUE_ALL = 7
CHUNK = 64


class gdr_problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("Hk", ctypes.c_int), ("Hv", ctypes.c_int),
                ("DK", ctypes.c_int), ("DV", ctypes.c_int), ("num_seqs", ctypes.c_int),
                ("cu_seqlens", ctypes.c_void_p), ("dtype", ctypes.c_int), ("layout", ctypes.c_int),
                ("scale", ctypes.c_float), ("h_dtype", ctypes.c_int), ("prologue", ctypes.c_uint),
                ("save_wy", ctypes.c_int), ("cp_fwd", ctypes.c_int), ("cp_bwd", ctypes.c_int)]


class GDRError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib_handle().gdr_status_string(status).decode() if _LIB is not None else str(status)
        if status == GDR_ERR_CUDA and _LIB is not None:
            ce = _LIB.gdr_debug_last_cuda_error()
            msg += f" ({_LIB.gdr_debug_cuda_error_string(ce).decode()}, cudaError {ce})"
        super().__init__(f"{where}: {msg}")


_LIB = None
_STAGE_ARR = None

EXPORTS = ["gdr_max_chunks", "gdr_saved_states_bytes", "gdr_fwd_workspace_bytes", "gdr_bwd_workspace_bytes",
           "gdr_fwd", "gdr_bwd", "gdr_workspace_status", "gdr_status_string", "gdr_path",
           "gdr_debug_set_stage_events", "gdr_debug_stage_count", "gdr_debug_stage_name",
           "gdr_debug_launch_count", "gdr_debug_last_cuda_error", "gdr_debug_cuda_error_string", "gdr_fwd_noalloc", "gdr_noalloc_status", "gdr_debug_tc_gemm", "gdr_debug_timeout_selftest", "gdr_debug_cp_segment", "gdr_debug_cp_segments"]


def _open(path: str):
    """dlopen one build of the library and declare its entry points' C signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(gdr_problem)
    vp, sz, i, u32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.POINTER(ctypes.c_uint32)
    for name in ["gdr_max_chunks", "gdr_saved_states_bytes", "gdr_fwd_workspace_bytes",
                 "gdr_bwd_workspace_bytes"]:
        getattr(lib, name).argtypes = [P]
        getattr(lib, name).restype = sz
    lib.gdr_path.argtypes = [P]
    lib.gdr_path.restype = i
    lib.gdr_fwd.argtypes = [P] + [vp] * 9 + [vp, sz, vp]
    lib.gdr_fwd.restype = i
    lib.gdr_bwd.argtypes = [P] + [vp] * 14 + [vp, sz, vp]
    lib.gdr_bwd.restype = i
    lib.gdr_fwd_noalloc.argtypes = [P] + [vp] * 9 + [vp]
    lib.gdr_fwd_noalloc.restype = i
    lib.gdr_noalloc_status.argtypes = [vp, u32p]
    lib.gdr_noalloc_status.restype = i
    lib.gdr_workspace_status.argtypes = [vp, vp, u32p]
    lib.gdr_workspace_status.restype = i
    lib.gdr_status_string.argtypes = [i]
    lib.gdr_status_string.restype = ctypes.c_char_p
    lib.gdr_debug_set_stage_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), i]
    lib.gdr_debug_set_stage_events.restype = None
    lib.gdr_debug_stage_count.argtypes = []
    lib.gdr_debug_stage_count.restype = i
    lib.gdr_debug_stage_name.argtypes = [i]
    lib.gdr_debug_stage_name.restype = ctypes.c_char_p
    lib.gdr_debug_launch_count.argtypes = []
    lib.gdr_debug_launch_count.restype = ctypes.c_ulonglong
    lib.gdr_debug_last_cuda_error.argtypes = []
    lib.gdr_debug_last_cuda_error.restype = i
    lib.gdr_debug_cuda_error_string.argtypes = [i]
    lib.gdr_debug_cuda_error_string.restype = ctypes.c_char_p
    lib.gdr_debug_tc_gemm.argtypes = [vp, vp, vp, i, i, i, i, vp, vp]
    lib.gdr_debug_tc_gemm.restype = i
    lib.gdr_debug_timeout_selftest.argtypes = [vp, ctypes.c_ulonglong, vp, vp]
    lib.gdr_debug_timeout_selftest.restype = i
    lib.gdr_debug_cp_segment.argtypes = [i, i, i, i, ctypes.POINTER(ctypes.c_int)]
    lib.gdr_debug_cp_segment.restype = i
    lib.gdr_debug_cp_segments.argtypes = [P, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
    lib.gdr_debug_cp_segments.restype = i
    return lib


def _lib_handle():
    """Load libgdr.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libgdr.so not built ({LIB_PATH}); run `python -m chunked_gated_delta_04_gb300.build`")
        _LIB = _open(LIB_PATH)
    return _LIB


class library:
    """Context manager: route every call of this module through another build of the library
    (e.g. the delay-injection build libgdr_delay.so) and restore the default one after."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _LIB
        self.saved = _lib_handle()
        _LIB = _open(self.path)
        return _LIB

    def __exit__(self, *exc):
        global _LIB
        _LIB = self.saved
        return False


def load():
    return _lib_handle()


# ------------------------------------------------------------------ marshalling helpers
def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(dtype):
    return GDR_DTYPE_BF16 if dtype == torch.bfloat16 else (GDR_DTYPE_F32 if dtype == torch.float32 else 99)


def make_problem(B, T, Hk, Hv, DK, DV, dtype, layout="KV", cu_seqlens=None, num_seqs=None, scale=None,
                 h_dtype=torch.float32, prologue=0, save_wy=False, cp_fwd=1, cp_bwd=1):
    """Build a gdr_problem.  dtype, h_dtype (of h_saved): torch.float32/bfloat16; layout "KV"/"VK";
    prologue: bit set of GDR_PROLOGUE_* (the matching inputs are raw); save_wy: the forward keeps
    its chunk factors in the saved buffer for the backward; cp_fwd, cp_bwd: context-parallel
    segments per sequence of each direction (1: off, GDR_CP_AUTO: the library chooses)."""
    p = gdr_problem()
    p.B, p.T, p.Hk, p.Hv, p.DK, p.DV = B, T, Hk, Hv, DK, DV
    if cu_seqlens is not None:
        p.cu_seqlens = _ptr(cu_seqlens)
        p.num_seqs = (cu_seqlens.numel() - 1) if num_seqs is None else num_seqs
    else:
        p.cu_seqlens = None
        p.num_seqs = B if num_seqs is None else num_seqs
    p.dtype = _dtype_code(dtype)
    p.h_dtype = _dtype_code(h_dtype)
    p.prologue = int(prologue)
    p.save_wy = int(save_wy) if isinstance(save_wy, (bool, int)) else 99
    p.cp_fwd, p.cp_bwd = int(cp_fwd), int(cp_bwd)
    p.layout = {"KV": GDR_STATE_KV, "VK": GDR_STATE_VK}.get(layout, 99) if isinstance(layout, str) else layout
    p.scale = 0.0 if scale is None else float(scale)
    return p


def gdr_max_chunks(p) -> int:
    return _lib_handle().gdr_max_chunks(ctypes.byref(p))


def gdr_saved_states_bytes(p) -> int:
    return _lib_handle().gdr_saved_states_bytes(ctypes.byref(p))


def gdr_fwd_workspace_bytes(p) -> int:
    return _lib_handle().gdr_fwd_workspace_bytes(ctypes.byref(p))


def gdr_bwd_workspace_bytes(p) -> int:
    return _lib_handle().gdr_bwd_workspace_bytes(ctypes.byref(p))


def gdr_path(p) -> int:
    return _lib_handle().gdr_path(ctypes.byref(p))


def gdr_fwd(p, q, k, v, g, beta, S0, o, S_T, h_saved, workspace, workspace_bytes=None, stream=None) -> int:
    """C gdr_fwd on tensors / raw device pointers; returns the status code."""
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    return _lib_handle().gdr_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0),
                                 _ptr(o), _ptr(S_T), _ptr(h_saved), _ptr(workspace), wb, _stream_ptr(stream))


def gdr_bwd(p, q, k, v, g, beta, h_saved, dO, dS_T, dq, dk, dv, dg, dbeta, dS0, workspace,
            workspace_bytes=None, stream=None) -> int:
    """C gdr_bwd on tensors / raw device pointers; returns the status code."""
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    return _lib_handle().gdr_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                 _ptr(h_saved), _ptr(dO), _ptr(dS_T), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg),
                                 _ptr(dbeta), _ptr(dS0), _ptr(workspace), wb, _stream_ptr(stream))


def gdr_fwd_noalloc(p, q, k, v, g, beta, S0, o, S_T, h_saved, stream=None) -> int:
    """C gdr_fwd_noalloc (the forward with library-owned scratch, for callers that
    cannot allocate); returns the status code."""
    return _lib_handle().gdr_fwd_noalloc(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                         _ptr(S0), _ptr(o), _ptr(S_T), _ptr(h_saved), _stream_ptr(stream))


NOALLOC_MAX_WORKSPACE_BYTES = 64 << 20


def gdr_noalloc_status(stream=None):
    """Synchronises the stream; returns (status, raw flag bits) of gdr_fwd_noalloc's status word."""
    flags = ctypes.c_uint32(0)
    st = _lib_handle().gdr_noalloc_status(_stream_ptr(stream), ctypes.byref(flags))
    return st, flags.value


def gdr_workspace_status(workspace, stream=None):
    """Synchronises the stream; returns (status, raw flag bits)."""
    flags = ctypes.c_uint32(0)
    st = _lib_handle().gdr_workspace_status(_ptr(workspace), _stream_ptr(stream), ctypes.byref(flags))
    return st, flags.value


def gdr_status_string(s: int) -> str:
    return _lib_handle().gdr_status_string(s).decode()


def gdr_debug_set_stage_events(events) -> None:
    """events: list of torch.cuda.Event (created with enable_timing=True) or None to switch off."""
    lib = _lib_handle()
    if events is None:
        lib.gdr_debug_set_stage_events(None, 0)
        return
    global _STAGE_ARR
    for e in events:  # torch creates the cudaEvent_t handle lazily, at the first record
        e.record()
    torch.cuda.synchronize()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _STAGE_ARR = arr  # keep the handle array alive while the library may use it
    lib.gdr_debug_set_stage_events(arr, len(events))


def gdr_debug_stage_names() -> list:
    lib = _lib_handle()
    return [lib.gdr_debug_stage_name(i).decode() for i in range(lib.gdr_debug_stage_count())]


def gdr_debug_tc_gemm(A, B, D, N, K, a_mn, b_mn, status, stream=None) -> int:
    return _lib_handle().gdr_debug_tc_gemm(_ptr(A), _ptr(B), _ptr(D), N, K, a_mn, b_mn, _ptr(status),
                                           _stream_ptr(stream))


def gdr_debug_timeout_selftest(status, limit_ns, waited_ns, stream=None) -> int:
    return _lib_handle().gdr_debug_timeout_selftest(_ptr(status), int(limit_ns), _ptr(waited_ns),
                                                    _stream_ptr(stream))


def gdr_debug_cp_segment(c0: int, c1: int, P: int, s: int):
    """(first chunk, end chunk, number of segments) of context-parallel segment s (host only)."""
    out = (ctypes.c_int * 3)()
    st = _lib_handle().gdr_debug_cp_segment(c0, c1, P, s, out)
    if st != 0:
        raise ValueError(f"gdr_debug_cp_segment({c0}, {c1}, {P}, {s}): invalid arguments")
    return tuple(out)


def gdr_debug_cp_segments(p):
    """(forward, backward) segment counts a call with problem p would use (1: none)."""
    f, b = ctypes.c_int(0), ctypes.c_int(0)
    st = _lib_handle().gdr_debug_cp_segments(ctypes.byref(p), ctypes.byref(f), ctypes.byref(b))
    if st != 0:
        raise GDRError(st, "gdr_debug_cp_segments")
    return f.value, b.value


GDR_CP_AUTO = -1


def gdr_debug_launch_count() -> int:
    return _lib_handle().gdr_debug_launch_count()


def _check(st, where):
    if st != GDR_OK:
        raise GDRError(st, where)


def _problem_for(q, v, cu_seqlens, layout, scale, h_dtype=torch.float32, prologue=0, save_wy=False, cp_fwd=1,
                 cp_bwd=1):
    B, T, Hk, DK = q.shape
    Hv, DV = v.shape[2], v.shape[3]
    return make_problem(B, T, Hk, Hv, DK, DV, q.dtype, layout, cu_seqlens, scale=scale, h_dtype=h_dtype,
                        prologue=prologue, save_wy=save_wy, cp_fwd=cp_fwd, cp_bwd=cp_bwd)


def alloc_saved(p, h_dtype, device) -> torch.Tensor:
    """The saved buffer of problem p: a [max_chunks, Hv, DK, DV] h_dtype view of the chunk-start
    states whose storage also holds the saved factors when p.save_wy is set (the view starts at
    the buffer's first byte, so its data pointer is the buffer's)."""
    nbytes = gdr_saved_states_bytes(p)
    shape = (gdr_max_chunks(p), p.Hv, p.DK, p.DV)
    states = math.prod(shape) * torch.empty((), dtype=h_dtype).element_size()
    buf = torch.empty(max(nbytes, states), dtype=torch.uint8, device=device)
    return buf[:states].view(h_dtype).view(shape)


def _check_saved(p, h_saved):
    need = gdr_saved_states_bytes(p)
    have = h_saved.untyped_storage().nbytes() - h_saved.storage_offset() * h_saved.element_size()
    if have < need:
        raise ValueError(f"saved buffer holds {have} bytes, the problem needs {need} (save_wy={p.save_wy}): "
                         "allocate it with alloc_saved")


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    # torch's allocator returns 512-byte aligned blocks, which covers the 256-byte requirement
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ allocating helpers
def forward(q, k, v, g, beta, S0=None, cu_seqlens=None, layout="KV", scale=None, output_final_state=True,
            workspace=None, stream=None, h_dtype=torch.float32, prologue=0, save_wy=False, cp=1):
    """Run gdr_fwd; returns (o, S_T or None, h_saved).  h_dtype: dtype of h_saved; prologue:
    GDR_PROLOGUE_* bits (q, k, g, beta raw where set); save_wy: h_saved's storage also keeps the
    chunk factors, and backward() must be given save_wy=True too; cp: context-parallel segments
    per sequence (1: off)."""
    p = _problem_for(q, v, cu_seqlens, layout, scale, h_dtype, prologue, save_wy, cp_fwd=cp)
    dev = q.device
    N = p.num_seqs
    o = torch.empty_like(v)
    sshape = (N, p.Hv, p.DK, p.DV) if layout == "KV" else (N, p.Hv, p.DV, p.DK)
    S_T = torch.empty(sshape, dtype=torch.float32, device=dev) if output_final_state else None
    h_saved = alloc_saved(p, h_dtype, dev)
    if workspace is None:
        workspace = alloc_workspace(gdr_fwd_workspace_bytes(p), dev)
    _check(gdr_fwd(p, q, k, v, g, beta, S0, o, S_T, h_saved, workspace, stream=stream), "gdr_fwd")
    return o, S_T, h_saved


def backward(q, k, v, g, beta, h_saved, dO, dS_T=None, cu_seqlens=None, layout="KV", scale=None,
             want_dS0=True, workspace=None, stream=None, prologue=0, save_wy=False, cp=1):
    """Run gdr_bwd; returns (dq, dk, dv, dg, dbeta, dS0 or None).  h_saved's dtype selects h_dtype;
    with prologue bits the gradients are w.r.t. the raw inputs; save_wy as given to forward(); cp:
    context-parallel segments per sequence (1: off; independent of the forward's)."""
    p = _problem_for(q, v, cu_seqlens, layout, scale, h_saved.dtype, prologue, save_wy, cp_bwd=cp)
    _check_saved(p, h_saved)
    dev = q.device
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dg = torch.empty_like(g)
    dbeta = torch.empty_like(beta)
    N = p.num_seqs
    sshape = (N, p.Hv, p.DK, p.DV) if layout == "KV" else (N, p.Hv, p.DV, p.DK)
    dS0 = torch.empty(sshape, dtype=torch.float32, device=dev) if want_dS0 else None
    if workspace is None:
        workspace = alloc_workspace(gdr_bwd_workspace_bytes(p), dev)
    _check(gdr_bwd(p, q, k, v, g, beta, h_saved, dO, dS_T, dq, dk, dv, dg, dbeta, dS0, workspace, stream=stream),
           "gdr_bwd")
    return dq, dk, dv, dg, dbeta, dS0


class _GDRFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, g, beta, S0, cu_seqlens, layout, scale, h_dtype, prologue, save_wy, cp_fwd, cp_bwd):
        o, S_T, h_saved = forward(q, k, v, g, beta, S0, cu_seqlens, layout, scale, h_dtype=h_dtype,
                                  prologue=prologue, save_wy=save_wy, cp=cp_fwd)
        ctx.save_for_backward(q, k, v, g, beta, h_saved, cu_seqlens)
        ctx.layout, ctx.scale, ctx.has_S0, ctx.prologue = layout, scale, S0 is not None, prologue
        ctx.save_wy, ctx.cp_bwd = save_wy, cp_bwd
        return o, S_T

    @staticmethod
    def backward(ctx, do, dS_T):
        q, k, v, g, beta, h_saved, cu_seqlens = ctx.saved_tensors
        dq, dk, dv, dg, dbeta, dS0 = backward(q, k, v, g, beta, h_saved, do.contiguous(),
                                              None if dS_T is None else dS_T.contiguous(), cu_seqlens,
                                              ctx.layout, ctx.scale, want_dS0=ctx.has_S0, prologue=ctx.prologue,
                                              save_wy=ctx.save_wy, cp=ctx.cp_bwd)
        return dq, dk, dv, dg, dbeta, dS0, None, None, None, None, None, None, None, None


def chunk_gated_delta_rule(q, k, v, g, beta, initial_state=None, cu_seqlens=None, layout="KV", scale=None,
                           h_dtype=torch.float32, prologue=0, save_wy=True, cp_fwd=1, cp_bwd=1):
    """Autograd entry point: returns (o, final_state).  Tensors as in include/gdr.h; h_dtype is the
    dtype of the chunk-start states kept for the backward (bfloat16 halves their memory); prologue
    (GDR_PROLOGUE_* bits) makes the operator normalise q, k and map raw gate / beta logits itself;
    save_wy (default) keeps the forward's chunk factors for the backward (49408 bytes per chunk and
    v-head more saved memory, no recomputation in the backward; same results bit for bit); cp_fwd,
    cp_bwd: context-parallel segments per sequence of each direction (1: off), for few long
    sequences whose (sequence, v-head) chains would leave most SMs idle."""
    return _GDRFunction.apply(q, k, v, g, beta, initial_state, cu_seqlens, layout, scale, h_dtype, prologue,
                              save_wy, cp_fwd, cp_bwd)
