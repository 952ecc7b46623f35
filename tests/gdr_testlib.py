"""Shared helpers for the GPU parity tests: run the CUDA path, run the oracle, compare."""
from __future__ import annotations

import numpy as np
import torch

import chunked_gated_delta_04_gb300 as gdr
import oracle

OUT_KEYS_FWD = ["o", "S_T", "h_saved"]
OUT_KEYS_BWD = ["dq", "dk", "dv", "dg", "dbeta", "dS0"]


def tol_for(dtype) -> float:
    """max|got - ref| / max|ref| bound per output tensor: 1e-4 for fp32 inputs, 2e-2 for bf16."""
    return 1e-4 if dtype == torch.float32 else 2e-2


def to_device(inp: dict, dev="cuda") -> dict:
    out = {}
    for k_, v_ in inp.items():
        out[k_] = v_.to(dev) if isinstance(v_, torch.Tensor) else v_
    return out


def run_gpu(inp: dict, backward: bool = True, stream=None, h_dtype=torch.float32, prologue=0,
            save_wy=False) -> dict:
    """Run gdr_fwd (+ gdr_bwd) on device copies of ``inp``; returns device tensors."""
    d = to_device(inp)
    layout = inp["layout"]
    o, S_T, h_saved = gdr.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S0"], d["cu_seqlens"], layout,
                                  stream=stream, h_dtype=h_dtype, prologue=prologue, save_wy=save_wy)
    res = {"o": o, "S_T": S_T, "h_saved": h_saved}
    if backward:
        dq, dk, dv, dg, dbeta, dS0 = gdr.backward(d["q"], d["k"], d["v"], d["g"], d["beta"], h_saved, d["dO"],
                                                  d["dS_T"], d["cu_seqlens"], layout, stream=stream,
                                                  prologue=prologue, save_wy=save_wy)
        res.update(dq=dq, dk=dk, dv=dv, dg=dg, dbeta=dbeta, dS0=dS0)
    return res


def to_np(t) -> np.ndarray:
    return t.detach().float().double().cpu().numpy()


def relmax(got, ref) -> float:
    den = np.abs(ref).max() if ref.size else 0.0
    num = np.abs(got - ref).max() if ref.size else 0.0
    if den == 0.0:
        return float(num)
    return float(num / den)


def compare(res: dict, ref: dict, tol: float, keys=None, n_chunks=None) -> dict:
    """rel_max per tensor; raises AssertionError listing every tensor above ``tol``."""
    keys = keys or [k_ for k_ in OUT_KEYS_FWD + OUT_KEYS_BWD if k_ in res and k_ in ref]
    errs = {}
    for key in keys:
        got = to_np(res[key])
        want = ref[key]
        if key == "h_saved":
            nc = want.shape[0] if n_chunks is None else n_chunks
            got = got[:nc]
        assert got.shape == want.shape, (key, got.shape, want.shape)
        assert np.isfinite(got).all(), f"{key}: non-finite values"
        errs[key] = relmax(got, want)
    bad = {k_: v_ for k_, v_ in errs.items() if not v_ <= tol}
    assert not bad, f"rel_max above {tol}: {bad} (all: {errs})"
    return errs


def head_slice(inp: dict, qk_heads) -> dict:
    """Restrict a workload to the given q/k heads and their v-heads (for sampled oracle checks)."""
    Hk = inp["q"].shape[2]
    Hv = inp["v"].shape[2]
    G = Hv // Hk
    vh = [i * G + jj for i in qk_heads for jj in range(G)]
    out = dict(inp)
    out["q"] = inp["q"][:, :, qk_heads]
    out["k"] = inp["k"][:, :, qk_heads]
    for key in ["v", "dO"]:
        out[key] = inp[key][:, :, vh]
    for key in ["g", "beta"]:
        out[key] = inp[key][:, :, vh]
    for key in ["S0", "dS_T"]:
        if inp[key] is not None:
            out[key] = inp[key][:, vh]
    return out, vh


def slice_result(res: dict, qk_heads, vh) -> dict:
    out = {}
    for key, t in res.items():
        if t is None:
            continue
        if key in ("dq", "dk"):
            out[key] = t[:, :, qk_heads]
        elif key in ("o", "dv", "dg", "dbeta"):
            out[key] = t[:, :, vh]
        elif key in ("S_T", "dS0", "h_saved"):
            out[key] = t[:, vh]
    return out


def reference(inp: dict, backward=True, prologue=0) -> dict:
    if prologue:
        from oracle import prologue as pl

        return pl.reference_with_prologue(inp, inp["layout"], prologue, backward=backward)
    return oracle.reference(inp, inp["layout"], backward=backward)
