"""gdr_fwd_noalloc: the forward for callers that cannot allocate device memory.

Some callers cannot pass the library a workspace and cannot allocate one: a plugin
whose host framework owns all device memory, or a latency-critical loop where a
cudaMalloc (which may synchronise the device) is not allowed.  For them the library
offers gdr_fwd_noalloc, whose scratch is a fixed array the library owns.  These
tests call it through the C ABI and check that it returns what gdr_fwd returns,
on two calls in a row with different inputs (so stale contents of the shared array
from the first call cannot leak into the second), and that an oversized problem is
refused before anything runs.

This file is collected last on purpose: a run that stops at the first failure has
then already run every other test.
"""
import pytest
import torch

import chunked_gated_delta_04_gb300 as gdr
from chunked_gated_delta_04_gb300.inputs import make_inputs, small_workload
from gdr_testlib import relmax, to_np, tol_for


def _run_both(w):
    inp = make_inputs(w)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    B, T, Hk, DK = d["q"].shape
    Hv, DV = d["v"].shape[2], d["v"].shape[3]
    p = gdr.make_problem(B, T, Hk, Hv, DK, DV, d["q"].dtype, w.layout, d["cu_seqlens"])
    assert gdr.gdr_fwd_workspace_bytes(p) <= gdr.NOALLOC_MAX_WORKSPACE_BYTES
    N = p.num_seqs
    sshape = (N, Hv, DK, DV) if w.layout == "KV" else (N, Hv, DV, DK)
    outs = []
    for use_noalloc in (False, True):
        o = torch.full_like(d["v"], float("nan"))
        S_T = torch.full(sshape, float("nan"), device="cuda")
        h = torch.full((gdr.gdr_max_chunks(p), Hv, DK, DV), float("nan"), device="cuda")
        if use_noalloc:
            st = gdr.gdr_fwd_noalloc(p, d["q"], d["k"], d["v"], d["g"], d["beta"], d["S0"], o, S_T, h)
        else:
            ws = gdr.alloc_workspace(gdr.gdr_fwd_workspace_bytes(p), "cuda")
            st = gdr.gdr_fwd(p, d["q"], d["k"], d["v"], d["g"], d["beta"], d["S0"], o, S_T, h, ws)
        assert st == gdr.GDR_OK, gdr.gdr_status_string(st)
        torch.cuda.synchronize()
        outs.append({"o": o, "S_T": S_T, "h_saved": h})
    return outs


@pytest.mark.gpu
def test_noalloc_forward_matches_gdr_fwd_on_two_calls_in_a_row():
    tol = tol_for(torch.bfloat16)
    for seed, T in ((0, 300), (1, 190)):
        w = small_workload(f"noalloc{seed}", torch.bfloat16, B=1, T=T, Hk=1, Hv=2, DK=128, DV=128, seed=seed)
        ref, got = _run_both(w)
        for key in ("o", "S_T", "h_saved"):
            a, b = to_np(got[key]), to_np(ref[key])
            assert (a == a).all(), f"{key}: unwritten or non-finite values"
            assert relmax(a, b) <= tol, (seed, key, relmax(a, b))


def test_noalloc_refuses_problems_beyond_its_scratch():
    # host-side check, before any CUDA call: no GPU needed
    p = gdr.make_problem(4, 8192, 16, 32, 128, 128, torch.bfloat16, "KV")
    assert gdr.gdr_fwd_workspace_bytes(p) > gdr.NOALLOC_MAX_WORKSPACE_BYTES
    fake = 1 << 20
    st = gdr.gdr_fwd_noalloc(p, fake, fake, fake, fake, fake, None, fake, None, fake, stream=0)
    assert st == gdr.GDR_ERR_WORKSPACE
