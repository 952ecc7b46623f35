"""Failure detection without a GPU fault: bounded waits give up and report a status.

A kernel waits on an mbarrier that nothing completes, with a 20 ms limit: it must
return, set the timeout bit, and leave the context usable.  The workspace status word
is mapped to the right status codes.  Nothing here traps, faults or hangs a GPU.
"""
import pytest
import torch

import chunked_gated_delta_04_gb300 as gdr

pytestmark = pytest.mark.gpu


def test_bounded_wait_expires_and_reports():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    assert gdr.gdr_debug_timeout_selftest(status, 20_000_000, waited) == 0
    torch.cuda.synchronize()
    assert status.item() & (1 << 1)
    assert 20_000_000 <= waited.item() < 1_000_000_000
    # the context is still usable
    x = torch.ones(1024, device="cuda")
    assert float(x.sum()) == 1024.0


def test_workspace_status_word_maps_to_status_codes():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert gdr.gdr_workspace_status(ws)[0] == gdr.GDR_OK
    ws.view(torch.int32)[0] = 1 << 1  # a kernel's bounded wait ran out
    st, flags = gdr.gdr_workspace_status(ws)
    assert st == gdr.GDR_ERR_TIMEOUT and flags == 2
    ws.view(torch.int32)[0] = 1  # malformed cu_seqlens seen by the index kernel
    assert gdr.gdr_workspace_status(ws)[0] == gdr.GDR_ERR_INVALID_ARG


def test_malformed_cu_seqlens_is_reported_not_computed():
    import torch

    from chunked_gated_delta_04_gb300.inputs import make_inputs, small_workload

    w = small_workload("bad", torch.bfloat16, Hk=1, Hv=1, DK=128, DV=128, seqlens=[70, 60])
    inp = make_inputs(w)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    d["cu_seqlens"] = torch.tensor([0, 90, 80], dtype=torch.int32, device="cuda")  # decreasing
    p = gdr.make_problem(1, 130, 1, 1, 128, 128, torch.bfloat16, "KV", d["cu_seqlens"])
    ws = gdr.alloc_workspace(gdr.gdr_fwd_workspace_bytes(p), "cuda")
    o = torch.zeros_like(d["v"])
    h = torch.zeros((gdr.gdr_max_chunks(p), 1, 128, 128), device="cuda")
    st = gdr.gdr_fwd(p, d["q"], d["k"], d["v"], d["g"], d["beta"], None, o, None, h, ws)
    assert st == gdr.GDR_OK  # launched: the host never reads cu_seqlens
    assert gdr.gdr_workspace_status(ws)[0] == gdr.GDR_ERR_INVALID_ARG
    assert float(o.abs().sum()) == 0.0  # nothing computed
