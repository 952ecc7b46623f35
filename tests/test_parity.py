"""GPU parity: the CUDA path against the fp64 oracle, element by element.

Bar: max|got - ref| / max|ref| per output tensor (o, S_T, h_saved, dq, dk, dv, dg,
dbeta, dS0) <= 1e-4 for fp32 inputs and <= 2e-2 for bf16 inputs; the oracle runs on
the exact (rounded) inputs the GPU sees.  Small cases span several chunks and a
ragged tail; the named full-size workloads are checked on sampled heads (all
tokens, all chunks of the sampled heads) in the same launch configuration the
benchmark times.
"""
import numpy as np
import pytest
import torch

import chunked_gated_delta_04_gb300 as gdr
from chunked_gated_delta_04_gb300.inputs import WORKLOADS, make_inputs, small_workload
from gdr_testlib import (OUT_KEYS_BWD, OUT_KEYS_FWD, compare, head_slice, record_margins, reference, run_gpu,
                         slice_result, to_device, tol_for)

pytestmark = pytest.mark.gpu


def _check(w, heads=None, ref=None, **run_kw):
    inp = make_inputs(w)
    res = run_gpu(inp, **run_kw)
    torch.cuda.synchronize()
    if heads is not None:
        sub, vh = head_slice(inp, heads)
        ref = reference(sub) if ref is None else ref
        res = slice_result(res, heads, vh)
    else:
        ref = reference(inp) if ref is None else ref
    return compare(res, ref, tol_for(w.dtype))


SMALL = [
    # name, dtype, B, T, Hk, Hv, D, layout, S0, dST
    ("f32_t1", torch.float32, 1, 1, 1, 1, 32, "KV", True, True),
    ("f32_t63", torch.float32, 1, 63, 1, 1, 64, "KV", False, False),
    ("f32_t64", torch.float32, 2, 64, 1, 1, 16, "VK", True, True),
    ("f32_t65", torch.float32, 1, 65, 1, 2, 32, "KV", True, True),
    ("f32_t130_gva", torch.float32, 2, 130, 2, 4, 32, "VK", True, False),
    ("f32_d128", torch.float32, 1, 200, 1, 1, 128, "KV", True, True),
    ("bf16_t129", torch.bfloat16, 1, 129, 1, 1, 128, "KV", True, True),
    ("bf16_t300_b2", torch.bfloat16, 2, 300, 2, 2, 128, "VK", True, True),
    ("bf16_gva", torch.bfloat16, 1, 192, 1, 2, 128, "KV", False, False),
    ("bf16_d64", torch.bfloat16, 1, 100, 1, 1, 64, "KV", True, True),
    # more state CTAs (sequences x v-heads x 4) than SMs: the single-buffered state kernel
    ("bf16_many_ctas", torch.bfloat16, 3, 200, 13, 13, 128, "KV", True, True),
    ("bf16_many_ctas_gva", torch.bfloat16, 1, 200, 10, 40, 128, "VK", True, False),
]


@pytest.mark.parametrize("dt,D", [(torch.float32, 32), (torch.bfloat16, 128)])
def test_strong_decay_gates(dt, D):
    # g = logsigmoid(N(-4, 1)) ~ -4 per token: in-chunk cumsums reach ~ -250, so any
    # exp(gamma_r - gamma_s) evaluated above the diagonal would overflow to inf
    _check(small_workload("strong_decay", dt, B=1, T=192, Hk=1, Hv=1, DK=D, DV=D, g_shift=-4.0))


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_shapes(case):
    name, dt, B, T, Hk, Hv, D, layout, s0, dst = case
    _check(small_workload(name, dt, B, T, Hk, Hv, D, D, layout, s0, dst))


@pytest.mark.parametrize("dt,D", [(torch.float32, 32), (torch.bfloat16, 128)])
def test_varlen_ragged(dt, D):
    # lengths: empty, 1, exactly one chunk, a ragged tail, several chunks
    w = small_workload("varlen", dt, Hk=1, Hv=2, DK=D, DV=D, seqlens=[0, 1, 64, 77, 200], layout="VK")
    _check(w)


def test_tiny_fp32_workload():
    _check(WORKLOADS["tiny_fp32"])


# The named workloads at full size, on sampled heads (every token and chunk of those heads), in
# each mode the benchmark can run: the backward recomputing the chunk factors, the forward
# saving them (the benchmark's default), and (b2_t4096) bf16 chunk-start states.  Each case's
# per-tensor rel_max is recorded in the parity-margins table (see gdr_testlib.record_margins).
NAMED = [("tiny_fp32", None, "simt", {}),
         ("tiny_fp32", None, "simt, saved", {"save_wy": True}),
         ("b2_t4096", [0, 15], "recompute", {}),
         ("b2_t4096", [0, 15], "saved", {"save_wy": True}),
         ("b2_t4096", [0, 15], "saved, h bf16", {"save_wy": True, "h_dtype": torch.bfloat16}),
         ("varlen8", [3], "recompute", {}),
         ("varlen8", [3], "saved", {"save_wy": True}),
         ("varlen8", [3], "recompute, cp 3/5", {"cp_fwd": 3, "cp_bwd": 5}),
         ("long_t65536", [7], "recompute", {}),
         ("long_t65536", [7], "saved", {"save_wy": True}),
         ("long_t65536", [7], "saved, cp 8/8", {"save_wy": True, "cp_fwd": 8, "cp_bwd": 8}),
         ("gva_b4_t8192", [0], "recompute", {}),
         ("gva_b4_t8192", [0], "saved", {"save_wy": True}),
         ("gva_b4_t8192", [0], "saved, cp 4/4", {"save_wy": True, "cp_fwd": 4, "cp_bwd": 4})]
_REF_CACHE = {}


@pytest.mark.slow
@pytest.mark.parametrize("name,heads,mode,kw", NAMED, ids=[f"{c[0]}-{c[2].replace(', ', '-').replace(' ', '_')}"
                                                            for c in NAMED])
def test_named_workloads_sampled_heads(name, heads, mode, kw):
    w = WORKLOADS[name]
    key = (name, tuple(heads) if heads else None)
    if key not in _REF_CACHE:  # the oracle's answer does not depend on the mode: compute it once
        _REF_CACHE.clear()
        inp = make_inputs(w)
        _REF_CACHE[key] = reference(head_slice(inp, heads)[0] if heads else inp)
    errs = _check(w, heads, ref=_REF_CACHE[key], **kw)
    record_margins(name, mode, "all" if heads is None else ",".join(map(str, heads)), errs, tol_for(w.dtype))


def test_varlen_matches_separate_fixed_length_runs():
    """Packing sequences with cu_seqlens gives bitwise the same results as separate runs."""
    lens = [70, 130]
    w = small_workload("vl", torch.bfloat16, Hk=1, Hv=1, DK=128, DV=128, seqlens=lens)
    inp = make_inputs(w)
    res = run_gpu(inp)
    cu = [0, 70, 200]
    for n, L in enumerate(lens):
        sub = dict(inp)
        for key in ["q", "k", "v", "dO", "g", "beta"]:
            sub[key] = inp[key][:, cu[n]:cu[n + 1]].contiguous()
        for key in ["S0", "dS_T"]:
            sub[key] = inp[key][n:n + 1].contiguous()
        sub["cu_seqlens"] = None
        r1 = run_gpu(sub)
        for key in ["o", "dq", "dk", "dv", "dg", "dbeta"]:
            assert torch.equal(r1[key], res[key][:, cu[n]:cu[n + 1]]), key
        for key in ["S_T", "dS0"]:
            assert torch.equal(r1[key][0], res[key][n]), key


def test_null_states_equal_zero_states():
    w = small_workload("z", torch.bfloat16, T=150, DK=128, DV=128, with_S0=False, with_dST=False)
    inp = make_inputs(w)
    r0 = run_gpu(inp)
    inp2 = dict(inp)
    inp2["S0"] = torch.zeros(1, 1, 128, 128)
    inp2["dS_T"] = torch.zeros(1, 1, 128, 128)
    r1 = run_gpu(inp2)
    for key in r0:
        if r0[key] is not None:
            assert torch.equal(r0[key], r1[key]), key


def test_kv_and_vk_layouts_are_transposes():
    w = small_workload("kv", torch.bfloat16, T=140, DK=128, DV=128, layout="KV")
    inp = make_inputs(w)
    rk = run_gpu(inp)
    inp2 = dict(inp)
    inp2["layout"] = "VK"
    inp2["S0"] = inp["S0"].transpose(-1, -2).contiguous()
    inp2["dS_T"] = inp["dS_T"].transpose(-1, -2).contiguous()
    rv = run_gpu(inp2)
    for key in ["o", "h_saved", "dq", "dk", "dv", "dg", "dbeta"]:
        assert torch.equal(rk[key], rv[key]), key
    assert torch.equal(rk["S_T"], rv["S_T"].transpose(-1, -2))
    assert torch.equal(rk["dS0"], rv["dS0"].transpose(-1, -2))


def test_runs_are_bitwise_deterministic():
    w = small_workload("det", torch.bfloat16, B=2, T=257, Hk=1, Hv=2, DK=128, DV=128)
    inp = make_inputs(w)
    r1, r2 = run_gpu(inp), run_gpu(inp)
    for key in r1:
        if r1[key] is not None:
            assert torch.equal(r1[key], r2[key]), key


def test_autograd_function_matches_oracle():
    import chunked_gated_delta_04_gb300 as gdr

    w = small_workload("ag", torch.bfloat16, T=100, DK=128, DV=128)
    inp = make_inputs(w)
    dev = {k_: (v_.cuda() if isinstance(v_, torch.Tensor) else v_) for k_, v_ in inp.items()}
    leaves = {k_: dev[k_].clone().requires_grad_(True) for k_ in ["q", "k", "v", "g", "beta", "S0"]}
    o, ST = gdr.chunk_gated_delta_rule(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["beta"],
                                       leaves["S0"], None, "KV")
    loss = (o.float() * dev["dO"].float()).sum() + (ST * dev["dS_T"]).sum()
    loss.backward()
    ref = reference(inp)
    got = {"o": o, "S_T": ST, "dq": leaves["q"].grad, "dk": leaves["k"].grad, "dv": leaves["v"].grad,
           "dg": leaves["g"].grad, "dbeta": leaves["beta"].grad, "dS0": leaves["S0"].grad}
    compare(got, ref, tol_for(torch.bfloat16))


def test_tensor_core_path_is_selected_for_bf16_d128():
    import chunked_gated_delta_04_gb300 as gdr

    p = gdr.make_problem(2, 4096, 16, 16, 128, 128, torch.bfloat16, "KV")
    assert gdr.gdr_path(p) == 1
    p32 = gdr.make_problem(1, 128, 1, 1, 64, 64, torch.float32, "KV")
    assert gdr.gdr_path(p32) == 0


# ---------------------------------------------------------------- bf16 saved chunk states
# h_saved rounded to bf16 (half the bytes of the largest tensor).  The backward reads
# the rounded states, and the SIMT forward computes o from them, so every output is
# held to the bf16 bar (2e-2) whatever the input dtype.
H_BF16_CASES = [
    # name, dtype, B, T, Hk, Hv, D, layout, seqlens
    ("tc_b2_t300", torch.bfloat16, 2, 300, 2, 2, 128, "VK", None),
    ("tc_gva_varlen", torch.bfloat16, 1, None, 1, 2, 128, "KV", [0, 1, 64, 77, 200]),
    ("simt_bf16_d64", torch.bfloat16, 1, 150, 1, 1, 64, "KV", None),
    ("simt_f32_d32", torch.float32, 2, 130, 2, 4, 32, "VK", None),
]


@pytest.mark.parametrize("case", H_BF16_CASES, ids=[c[0] for c in H_BF16_CASES])
def test_bf16_saved_states_match_oracle(case):
    name, dt, B, T, Hk, Hv, D, layout, lens = case
    if lens is None:
        w = small_workload(name, dt, B, T, Hk, Hv, D, D, layout)
    else:
        w = small_workload(name, dt, Hk=Hk, Hv=Hv, DK=D, DV=D, seqlens=lens, layout=layout)
    inp = make_inputs(w)
    res = run_gpu(inp, h_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert res["h_saved"].dtype == torch.bfloat16
    compare(res, reference(inp), 2e-2)


SAVE_WY_CASES = [
    # name, B, T, Hk, Hv, layout, seqlens, h_dtype, prologue, input dtype, D
    ("fused_b2_t300_vk", 2, 300, 2, 2, "VK", None, torch.float32, 0, torch.bfloat16, 128),  # fused walk + grad
    ("pair_varlen", 1, None, 1, 2, "KV", [0, 1, 64, 77, 200], torch.float32, 0, torch.bfloat16, 128),  # clusters
    ("group4_t130", 1, 130, 1, 4, "KV", None, torch.bfloat16, 0, torch.bfloat16, 128),  # group partials
    ("fused_prologue", 2, 193, 2, 2, "KV", None, torch.float32, 7, torch.bfloat16, 128),  # raw inputs
    # the SIMT path for heads of at most 64 features (fp32 factors in the saved buffer)
    ("simt_f32_b2_t130", 2, 130, 2, 2, "KV", None, torch.float32, 0, torch.float32, 64),
    ("simt_f32_varlen_gva", 1, None, 1, 2, "VK", [0, 1, 64, 77, 200], torch.float32, 0, torch.float32, 32),
    ("simt_bf16_d48_prologue", 2, 193, 2, 2, "KV", None, torch.float32, 7, torch.bfloat16, 48),
]


@pytest.mark.parametrize("case", SAVE_WY_CASES, ids=[c[0] for c in SAVE_WY_CASES])
def test_saved_factors_give_identical_results(case):
    """save_wy only moves where the chunk factors come from (kept by the forward instead of
    recomputed by the backward, by the same code on the same inputs): every output is bitwise
    the same as without it, and the oracle agrees."""
    name, B, T, Hk, Hv, layout, lens, h_dtype, pro, dt, D = case
    if lens is None:
        w = small_workload(name, dt, B, T, Hk, Hv, D, D, layout)
    else:
        w = small_workload(name, dt, Hk=Hk, Hv=Hv, DK=D, DV=D, seqlens=lens, layout=layout)
    inp = make_inputs(w, raw=bool(pro))
    base = run_gpu(inp, h_dtype=h_dtype, prologue=pro)
    res = run_gpu(inp, h_dtype=h_dtype, prologue=pro, save_wy=True)
    torch.cuda.synchronize()
    n_chunks = sum(-(-L // 64) for L in inp["seqlens"])  # slots past the real chunks stay unwritten
    for key in OUT_KEYS_FWD + OUT_KEYS_BWD:
        if base.get(key) is not None:
            a, b = (base[key], res[key]) if key != "h_saved" else (base[key][:n_chunks], res[key][:n_chunks])
            assert torch.equal(a, b), key
    compare(res, reference(inp, prologue=pro), 1e-4 if dt == torch.float32 else 2e-2)


def test_saved_factors_need_the_larger_buffer():
    w = small_workload("wyb", torch.bfloat16, 1, 130, 1, 1, 128, 128)
    inp = make_inputs(w)
    d = to_device(inp)
    _, _, hs = gdr.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S0"], None, "KV")
    with pytest.raises(ValueError):  # a states-only buffer cannot hold the factors
        gdr.backward(d["q"], d["k"], d["v"], d["g"], d["beta"], hs, d["dO"], d["dS_T"], None, "KV",
                     save_wy=True)


def test_bf16_saved_states_leave_tensor_core_forward_unchanged():
    """On the tensor-core path h_dtype only changes what is stored: o and S_T are bitwise
    the same, and the bf16 states are the fp32 states rounded to nearest even."""
    w = small_workload("hcmp", torch.bfloat16, B=2, T=257, Hk=1, Hv=2, DK=128, DV=128)
    inp = make_inputs(w)
    r32 = run_gpu(inp, backward=False)
    r16 = run_gpu(inp, backward=False, h_dtype=torch.bfloat16)
    assert torch.equal(r32["o"], r16["o"])
    assert torch.equal(r32["S_T"], r16["S_T"])
    assert torch.equal(r32["h_saved"].to(torch.bfloat16), r16["h_saved"])


# ---------------------------------------------------------------- fused input prologue
# Raw q, k (not normalised), raw gate and beta logits; the operator applies the q/k L2
# norm, logsigmoid and sigmoid itself and returns gradients w.r.t. the raw tensors.
PROLOGUE_CASES = [
    # name, dtype, B, T, Hk, Hv, D, layout, seqlens, flags
    ("tc_all", torch.bfloat16, 2, 300, 2, 2, 128, "KV", None, 7),
    ("tc_gva_varlen_all", torch.bfloat16, 1, None, 1, 2, 128, "VK", [0, 1, 64, 77, 200], 7),
    ("tc_qk_only", torch.bfloat16, 1, 150, 1, 1, 128, "KV", None, 1),
    ("tc_g_only", torch.bfloat16, 1, 150, 1, 1, 128, "KV", None, 2),
    ("tc_beta_only", torch.bfloat16, 1, 150, 1, 1, 128, "KV", None, 4),
    ("simt_f32_all", torch.float32, 2, 130, 2, 4, 32, "VK", None, 7),
    ("simt_bf16_d64_all", torch.bfloat16, 1, 150, 1, 1, 64, "KV", None, 7),
]


@pytest.mark.parametrize("case", PROLOGUE_CASES, ids=[c[0] for c in PROLOGUE_CASES])
def test_fused_prologue_matches_oracle(case):
    name, dt, B, T, Hk, Hv, D, layout, lens, flags = case
    if lens is None:
        w = small_workload(name, dt, B, T, Hk, Hv, D, D, layout)
    else:
        w = small_workload(name, dt, Hk=Hv // 2 if Hv > 1 else 1, Hv=Hv, DK=D, DV=D, seqlens=lens, layout=layout)
    inp = make_inputs(w, raw=True)
    # inputs whose prologue bit is off are passed already mapped
    if not flags & 1:
        for key in ["q", "k"]:
            inp[key] = torch.nn.functional.normalize(inp[key].float(), dim=-1).to(dt)
    if not flags & 2:
        inp["g"] = torch.nn.functional.logsigmoid(inp["g"])
    if not flags & 4:
        inp["beta"] = torch.sigmoid(inp["beta"].float()).to(dt)
    res = run_gpu(inp, prologue=flags)
    torch.cuda.synchronize()
    compare(res, reference(inp, prologue=flags), tol_for(dt))


def test_fused_prologue_autograd():
    import chunked_gated_delta_04_gb300 as gdr

    w = small_workload("agp", torch.bfloat16, T=100, DK=128, DV=128)
    inp = make_inputs(w, raw=True)
    dev = {k_: (v_.cuda() if isinstance(v_, torch.Tensor) else v_) for k_, v_ in inp.items()}
    leaves = {k_: dev[k_].clone().requires_grad_(True) for k_ in ["q", "k", "v", "g", "beta", "S0"]}
    o, ST = gdr.chunk_gated_delta_rule(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["beta"],
                                       leaves["S0"], None, "KV", prologue=gdr.GDR_PROLOGUE_ALL)
    loss = (o.float() * dev["dO"].float()).sum() + (ST * dev["dS_T"]).sum()
    loss.backward()
    ref = reference(inp, prologue=7)
    got = {"o": o, "S_T": ST, "dq": leaves["q"].grad, "dk": leaves["k"].grad, "dv": leaves["v"].grad,
           "dg": leaves["g"].grad, "dbeta": leaves["beta"].grad, "dS0": leaves["S0"].grad}
    compare(got, ref, tol_for(torch.bfloat16))


# ---------------------------------------------------------------- fused backward coverage
# Fixed-length tensor-core batches run the reverse walk and the gradients as one cooperative
# kernel.  These cases cover a CTA running several walk units (more (sequence, head, DV half)
# units than SMs), and Hv = 4 Hk (fp32 partials and the group reduce after the fused kernel).
@pytest.mark.parametrize("name,B,T,Hk,Hv", [("many_walk_units", 10, 130, 8, 8), ("gva4", 2, 150, 1, 4),
                                             ("few_chains_dv_halves", 1, 300, 2, 2)])
def test_fused_backward_shapes(name, B, T, Hk, Hv):
    import chunked_gated_delta_04_gb300 as gdr

    w = small_workload(name, torch.bfloat16, B=B, T=T, Hk=Hk, Hv=Hv, DK=128, DV=128)
    p = gdr.make_problem(B, T, Hk, Hv, 128, 128, torch.bfloat16, "KV")
    assert gdr.gdr_path(p) == 1
    _check(w)


# The walk runs as two DV halves per (sequence, v-head) while its units fill at most a quarter
# of the SMs (few chains: the walk is the critical path) and as one full-width unit otherwise.
# Full width through the stand-alone walk (cluster-pair gradients, Hv = 2 Hk, variable length)
# and through the fused kernel (fixed length), against the oracle.
@pytest.mark.parametrize("name,B,T,Hk,Hv,lens", [
    ("full_width_pair_varlen", 1, None, 4, 8, [0, 70, 130, 1, 200, 64]),
    ("full_width_fused", 3, 200, 8, 8, None),
])
def test_walk_full_width(name, B, T, Hk, Hv, lens):
    if lens is None:
        w = small_workload(name, torch.bfloat16, B=B, T=T, Hk=Hk, Hv=Hv, DK=128, DV=128)
    else:
        w = small_workload(name, torch.bfloat16, Hk=Hk, Hv=Hv, DK=128, DV=128, seqlens=lens)
    _check(w)
