"""GPU parity of intra-card context parallelism (FlashQLA PR #34, "Current status": intra-card CP,
with forward and backward segment counts set independently).

Each sequence is cut into segments at chunk boundaries; the first pass computes segment maps, a
scan chains the boundary states, and the second pass evaluates every segment from its true
boundary.  The results are the operator's own, so every case is compared with the fp64 oracle
(the plain recurrence) at the usual bars, over segment counts from 2 to more than a sequence's
chunk count, ragged tails, empty and one-token sequences, grouped v-heads (pair and partial
sums), both state layouts, bf16 saved states, saved chunk factors and slow decay.
"""
import pytest
import torch

import chunked_gated_delta_04_gb300 as gdr
from chunked_gated_delta_04_gb300.inputs import make_inputs, small_workload
from gdr_testlib import compare, reference, run_gpu, tol_for

pytestmark = pytest.mark.gpu

CASES = [
    # name, workload kwargs, run kwargs
    ("t841_p2", dict(B=1, T=841, Hk=2, Hv=2), dict(cp_fwd=2, cp_bwd=2)),
    ("t841_p3_p4", dict(B=1, T=841, Hk=2, Hv=2), dict(cp_fwd=3, cp_bwd=4)),
    ("t841_p5_p3_saved", dict(B=1, T=841, Hk=2, Hv=2), dict(cp_fwd=5, cp_bwd=3, save_wy=True)),
    # one segment per chunk, and more segments than chunks (clamped to the chunk count)
    ("t841_p14", dict(B=1, T=841, Hk=1, Hv=1), dict(cp_fwd=14, cp_bwd=14)),
    ("t841_p20", dict(B=1, T=841, Hk=1, Hv=1), dict(cp_fwd=20, cp_bwd=20)),
    ("b2_vk_pair", dict(B=2, T=500, Hk=1, Hv=2, layout="VK"), dict(cp_fwd=4, cp_bwd=4)),
    ("gva4_nostates", dict(B=1, T=700, Hk=1, Hv=4, with_S0=False, with_dST=False), dict(cp_fwd=3, cp_bwd=3)),
    ("varlen", dict(Hk=1, Hv=2, seqlens=[0, 1, 64, 77, 200, 900]), dict(cp_fwd=4, cp_bwd=6)),
    ("h_bf16_saved", dict(B=1, T=1000, Hk=1, Hv=2), dict(cp_fwd=4, cp_bwd=4, save_wy=True,
                                                         h_dtype=torch.bfloat16)),
    ("fwd_only_cp", dict(B=1, T=600, Hk=1, Hv=1), dict(cp_fwd=4, cp_bwd=1)),
    ("bwd_only_cp", dict(B=1, T=600, Hk=1, Hv=1), dict(cp_fwd=1, cp_bwd=4)),
    # slow decay (g = logsigmoid(N(2, 1)), the long-sequence workload's gates): the transitions
    # barely contract, so errors in them are not damped along the scan
    ("slow_decay_t4096_p8", dict(B=1, T=4096, Hk=1, Hv=1, layout="VK", g_shift=2.0), dict(cp_fwd=8, cp_bwd=8)),
    # very slow decay (g = logsigmoid(N(6, 1)), about -0.16 per chunk): the state remembers
    # across many segments, so the transitions and the scan carry most of each boundary state
    ("long_memory_t8192_p16", dict(B=1, T=8192, Hk=1, Hv=1, g_shift=6.0), dict(cp_fwd=16, cp_bwd=16)),
]


@pytest.mark.parametrize("name,wkw,rkw", CASES, ids=[c[0] for c in CASES])
def test_cp_matches_oracle(name, wkw, rkw):
    w = small_workload("cp_" + name, torch.bfloat16, DK=128, DV=128, **wkw)
    inp = make_inputs(w)
    res = run_gpu(inp, **rkw)
    torch.cuda.synchronize()
    compare(res, reference(inp), tol_for(w.dtype))


def test_cp_is_deterministic():
    """No float atomics and fixed summation orders: two runs agree bit for bit."""
    w = small_workload("cp_det", torch.bfloat16, B=1, T=1500, Hk=2, Hv=2, DK=128, DV=128)
    inp = make_inputs(w)
    r0 = run_gpu(inp, cp_fwd=5, cp_bwd=5)
    r1 = run_gpu(inp, cp_fwd=5, cp_bwd=5)
    for key, val in r0.items():
        if val is not None:
            assert torch.equal(val, r1[key]), key


def test_cp_close_to_single_chain():
    """Segmenting changes only rounding: the results stay within the bf16 bar of the plain chain's."""
    w = small_workload("cp_vs_chain", torch.bfloat16, B=1, T=2000, Hk=1, Hv=2, DK=128, DV=128)
    inp = make_inputs(w)
    base = run_gpu(inp)
    cp = run_gpu(inp, cp_fwd=6, cp_bwd=6)
    for key, val in base.items():
        if val is None:
            continue
        a, b = val.float(), cp[key].float()
        assert (a - b).abs().max().item() <= 2e-2 * a.abs().max().item(), key


def _auto_rule(chains, nc, backward, n_sm):
    """The documented GDR_CP_AUTO choice, restated."""
    if chains * 16 > n_sm:
        return 1
    P = min(32, nc // 16)
    while P >= 3 and ((chains * (1 + 2 * (P - 2)) > n_sm) if backward else (chains * (4 + 8 * (P - 2)) > 2 * n_sm)):
        P -= 1
    return P if P >= 3 else 1


@pytest.mark.parametrize("B,T,Hk,Hv", [(1, 65536, 2, 2), (1, 65536, 1, 1), (1, 8192, 1, 2), (1, 65536, 16, 16),
                                       (2, 4096, 16, 16), (1, 1000, 1, 1)])
def test_cp_auto_choice(B, T, Hk, Hv):
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    p = gdr.make_problem(B, T, Hk, Hv, 128, 128, torch.bfloat16, cp_fwd=gdr.GDR_CP_AUTO, cp_bwd=gdr.GDR_CP_AUTO)
    nc = (T + 63) // 64
    assert gdr.gdr_debug_cp_segments(p) == (_auto_rule(B * Hv, nc, False, n_sm), _auto_rule(B * Hv, nc, True, n_sm))


def test_cp_auto_matches_oracle():
    """GDR_CP_AUTO on one short chain (4 segments of 16 chunks each way) against the oracle."""
    w = small_workload("cp_auto", torch.bfloat16, B=1, T=4096, Hk=1, Hv=1, DK=128, DV=128)
    inp = make_inputs(w)
    p = gdr.make_problem(1, 4096, 1, 1, 128, 128, torch.bfloat16, cp_fwd=gdr.GDR_CP_AUTO, cp_bwd=gdr.GDR_CP_AUTO)
    assert gdr.gdr_debug_cp_segments(p) == (4, 4)
    res = run_gpu(inp, cp_fwd=gdr.GDR_CP_AUTO, cp_bwd=gdr.GDR_CP_AUTO)
    torch.cuda.synchronize()
    compare(res, reference(inp), tol_for(w.dtype))


def test_cp_with_fused_prologue():
    """Segments with raw inputs (q/k L2 norm, logsigmoid gate, sigmoid beta inside the operator)."""
    w = small_workload("cp_prologue", torch.bfloat16, B=1, T=900, Hk=1, Hv=2, DK=128, DV=128)
    inp = make_inputs(w, raw=True)
    res = run_gpu(inp, prologue=7, cp_fwd=4, cp_bwd=5, save_wy=True)
    torch.cuda.synchronize()
    compare(res, reference(inp, prologue=7), tol_for(w.dtype))


def _segment_scan_oracle(inp, P):
    """The contract's outputs from the fp64 segment-scan oracle (oracle/context_parallel.py) with P
    segments per sequence, in the layouts oracle.reference returns."""
    import numpy as np

    from oracle.context_parallel import cp_backward, cp_forward

    f = lambda t: None if t is None else t.detach().double().numpy()
    q, k, v, g, beta, dO = (f(inp[n]) for n in ("q", "k", "v", "g", "beta", "dO"))
    B, T, Hk, DK = q.shape
    Hv, DV = v.shape[2], v.shape[3]
    cu = inp["cu_seqlens"].numpy() if inp["cu_seqlens"] is not None else np.arange(B + 1) * T
    kv = inp["layout"] == "KV"
    to_S = lambda x: None if x is None else (np.swapaxes(x, -1, -2).copy() if kv else x)
    pk = lambda a: a.reshape(B * T, *a.shape[2:])
    scale = 1.0 / np.sqrt(DK)
    o, S_T, states = cp_forward(cu, Hk, Hv, scale, pk(q), pk(k), pk(v), pk(g), pk(beta), to_S(f(inp["S0"])), P)
    dq, dk, dv, dg, dbeta, dS0 = cp_backward(cu, Hk, Hv, scale, pk(q), pk(k), pk(v), pk(g), pk(beta),
                                             to_S(f(inp["S0"])), pk(dO), to_S(f(inp["dS_T"])), P)
    return {"o": o.reshape(B, T, Hv, DV), "S_T": to_S(S_T), "h_saved": np.swapaxes(states, -1, -2),
            "dq": dq.reshape(q.shape), "dk": dk.reshape(k.shape), "dv": dv.reshape(v.shape),
            "dg": dg.reshape(B, T, Hv), "dbeta": dbeta.reshape(B, T, Hv), "dS0": to_S(dS0)}


@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_cp_matches_segment_scan_oracle(P):
    """The GPU's segment passes against the fp64 segment-scan oracle with the same segment count,
    on ragged and empty sequences with grouped v-heads."""
    w = small_workload("cp_vs_scan_oracle", torch.bfloat16, Hk=1, Hv=2, DK=128, DV=128,
                       seqlens=[0, 77, 700, 1000], layout="VK")
    inp = make_inputs(w)
    res = run_gpu(inp, cp_fwd=P, cp_bwd=P, save_wy=True)
    torch.cuda.synchronize()
    compare(res, _segment_scan_oracle(inp, P), tol_for(w.dtype))
