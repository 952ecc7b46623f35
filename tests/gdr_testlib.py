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
            save_wy=False, cp_fwd=1, cp_bwd=1) -> dict:
    """Run gdr_fwd (+ gdr_bwd) on device copies of ``inp``; returns device tensors.  cp_fwd, cp_bwd:
    context-parallel segments per sequence of each direction (1: off)."""
    d = to_device(inp)
    layout = inp["layout"]
    o, S_T, h_saved = gdr.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S0"], d["cu_seqlens"], layout,
                                  stream=stream, h_dtype=h_dtype, prologue=prologue, save_wy=save_wy, cp=cp_fwd)
    res = {"o": o, "S_T": S_T, "h_saved": h_saved}
    if backward:
        dq, dk, dv, dg, dbeta, dS0 = gdr.backward(d["q"], d["k"], d["v"], d["g"], d["beta"], h_saved, d["dO"],
                                                  d["dS_T"], d["cu_seqlens"], layout, stream=stream,
                                                  prologue=prologue, save_wy=save_wy, cp=cp_bwd)
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


# ------------------------------------------------------------------ recorded parity margins
# The full-size parity tests record their per-tensor rel_max here; at the end of the session
# conftest.py merges them into a Markdown table (profiles/parity_margins.md by default, or the
# path in GDR_PARITY_MARGINS), one row per (workload, mode), so the margin against the bar is on
# record for every configuration the benchmark runs.
MARGIN_KEYS = ["o", "S_T", "h_saved", "dq", "dk", "dv", "dg", "dbeta", "dS0"]
_MARGINS: dict = {}


def record_margins(workload: str, mode: str, heads: str, errs: dict, tol: float) -> None:
    _MARGINS[(workload, mode)] = (heads, dict(errs), tol)


def _fmt(x) -> str:
    return "-" if x is None else f"{x:.2e}"


def write_margins(path: str, device_name: str) -> None:
    """Merge the recorded rows into the table at ``path`` (rows of other (workload, mode) pairs kept)."""
    import datetime
    import os

    if not _MARGINS:
        return
    rows = {}
    if os.path.exists(path):
        with open(path) as f:
            for line in f:
                cells = [c.strip() for c in line.strip().strip("|").split("|")]
                if line.startswith("| ") and len(cells) == len(MARGIN_KEYS) + 4 and cells[0] != "workload" \
                        and not cells[0].startswith("-"):
                    rows[(cells[0], cells[1])] = line.rstrip("\n")
    for (w, mode), (heads, errs, tol) in _MARGINS.items():
        worst = max((v for v in errs.values() if v is not None), default=0.0)
        cells = [w, mode, heads] + [_fmt(errs.get(k)) for k in MARGIN_KEYS] + [f"{tol:g} (worst/bar {worst / tol:.3f})"]
        rows[(w, mode)] = "| " + " | ".join(cells) + " |"
    head = ["# Parity margins of the full-size workloads against the fp64 oracle", "",
            "Written by `tests/test_parity.py::test_named_workloads_sampled_heads` "
            "(`python -m pytest tests -m gpu`); last update "
            f"{datetime.datetime.now(datetime.timezone.utc).strftime('%Y-%m-%d %H:%M UTC')} on {device_name}.",
            "Each cell is rel_max = max|got - ref| / max|ref| of one output tensor over the sampled heads",
            "(every token and chunk of those heads), oracle evaluated on the exact rounded inputs. Bar:",
            "2e-2 for bf16 inputs (and for bf16 saved states), 1e-4 for fp32 inputs. Modes: `recompute` =",
            "the backward recomputes the chunk factors; `saved` = the forward keeps them (the benchmark's",
            "mode); `h bf16` = bf16 chunk-start states; `cp f/b` = context-parallel segments per",
            "sequence, forward / backward. `-` = the workload has no such output.", "",
            "| workload | mode | heads | " + " | ".join(MARGIN_KEYS) + " | bar |",
            "|" + "---|" * (len(MARGIN_KEYS) + 4)]
    with open(path, "w") as f:
        f.write("\n".join(head + [rows[k] for k in sorted(rows)]) + "\n")
