"""gdr_fwd_noalloc: the forward for callers that cannot allocate device memory.

Some callers cannot pass the library a workspace and cannot allocate one: a plugin
whose host framework owns all device memory, or a latency-critical loop where a
cudaMalloc (which may synchronise the device) is not allowed.  For them the library
offers gdr_fwd_noalloc, whose scratch is a fixed array the library owns.  These
tests call it through the C ABI and check that it returns bit for bit what gdr_fwd
returns (the same kernels on the same inputs, only the scratch differs), on two calls
in a row with different inputs (so stale contents of the shared array from the first
call cannot leak into the second): on the tensor-core path (fixed length and
variable length, whose chunk tables live in the array) and on the fp32 SIMT path
(another scratch layout).  A malformed cu_seqlens must show up through
gdr_noalloc_status, and an oversized problem is refused before anything runs.

This file is collected last on purpose: a run that stops at the first failure has
then already run every other test.
"""
import pytest
import torch

import chunked_gated_delta_04_gb300 as gdr
from chunked_gated_delta_04_gb300.inputs import make_inputs, small_workload


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
            assert st == gdr.GDR_OK, gdr.gdr_status_string(st)
            assert gdr.gdr_noalloc_status()[0] == gdr.GDR_OK
        else:
            ws = gdr.alloc_workspace(gdr.gdr_fwd_workspace_bytes(p), "cuda")
            st = gdr.gdr_fwd(p, d["q"], d["k"], d["v"], d["g"], d["beta"], d["S0"], o, S_T, h, ws)
            assert st == gdr.GDR_OK, gdr.gdr_status_string(st)
        torch.cuda.synchronize()
        outs.append({"o": o, "S_T": S_T, "h_saved": h})
    return outs, sum(inp["seqlens"])


def _assert_same(w):
    (ref, got), n_tok = _run_both(w)
    for key in ("o", "S_T", "h_saved"):
        a, b = got[key], ref[key]
        if key == "h_saved":  # slots past the last real chunk are never written
            n = sum((L + 63) // 64 for L in make_inputs(w)["seqlens"])
            a, b = a[:n], b[:n]
        assert not torch.isnan(a).any(), f"{w.name} {key}: unwritten values"
        assert torch.equal(a, b), f"{w.name} {key}: differs from gdr_fwd"


@pytest.mark.gpu
def test_noalloc_forward_matches_gdr_fwd_on_two_calls_in_a_row():
    # tensor-core path, fixed length: two calls with different inputs and lengths
    for seed, T in ((0, 300), (1, 190)):
        _assert_same(small_workload(f"noalloc{seed}", torch.bfloat16, B=1, T=T, Hk=1, Hv=2, DK=128, DV=128,
                                    seed=seed))


@pytest.mark.gpu
def test_noalloc_varlen_and_fp32_paths_on_two_calls_in_a_row():
    # variable length (the chunk tables of the first call are in the array when the second runs)
    for seed, lens in ((2, [0, 70, 130, 1]), (3, [200, 64, 5])):
        _assert_same(small_workload(f"noalloc_vl{seed}", torch.bfloat16, Hk=1, Hv=2, DK=128, DV=128,
                                    seqlens=lens, layout="VK", seed=seed))
    # fp32 SIMT path, D = 64 (fp32 intermediates in the array)
    for seed, T in ((4, 128), (5, 77)):
        _assert_same(small_workload(f"noalloc_f32_{seed}", torch.float32, B=1, T=T, Hk=1, Hv=1, DK=64, DV=64,
                                    seed=seed))


@pytest.mark.gpu
def test_noalloc_reports_malformed_cu_seqlens():
    w = small_workload("noalloc_bad", torch.bfloat16, Hk=1, Hv=1, DK=128, DV=128, seqlens=[70, 60])
    inp = make_inputs(w)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    bad = torch.tensor([0, 90, 80], dtype=torch.int32, device="cuda")  # decreasing
    p = gdr.make_problem(1, 130, 1, 1, 128, 128, torch.bfloat16, "KV", bad)
    o = torch.zeros_like(d["v"])
    h = torch.zeros((gdr.gdr_max_chunks(p), 1, 128, 128), device="cuda")
    st = gdr.gdr_fwd_noalloc(p, d["q"], d["k"], d["v"], d["g"], d["beta"], None, o, None, h)
    assert st == gdr.GDR_OK  # launched: the host never reads cu_seqlens
    st, flags = gdr.gdr_noalloc_status()
    assert st == gdr.GDR_ERR_INVALID_ARG and flags & 1
    assert float(o.abs().sum()) == 0.0  # nothing computed
    # the next well-formed call clears the word again
    good = small_workload("noalloc_good", torch.bfloat16, Hk=1, Hv=1, DK=128, DV=128, seqlens=[70, 60])
    _assert_same(good)


def test_noalloc_refuses_problems_beyond_its_scratch():
    # host-side check, before any CUDA call: no GPU needed
    p = gdr.make_problem(4, 8192, 16, 32, 128, 128, torch.bfloat16, "KV")
    assert gdr.gdr_fwd_workspace_bytes(p) > gdr.NOALLOC_MAX_WORKSPACE_BYTES
    fake = 1 << 20
    st = gdr.gdr_fwd_noalloc(p, fake, fake, fake, fake, fake, None, fake, None, fake, stream=0)
    assert st == gdr.GDR_ERR_WORKSPACE
