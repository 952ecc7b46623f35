"""Pins for the fp64 oracle (CPU only).

The pages print no worked example and no numbers for the gated delta rule, so the
oracle is pinned to things other than itself:

* a hand-worked 2-token, 2x2 example (tests/golden/hand_2x2.json);
* central finite differences of L = <o, dO> + <S_T, dS_T> for every input;
* the closed form at beta = 0 (the state only decays: S_t = e^{Lambda_t} S0);
* the closed form of gated linear attention when the keys are orthonormal and S0 = 0
  (the erase term vanishes exactly);
* the exact-overwrite invariant S_t k_t = v_t for beta = 1 and unit keys (any gate);
* agreement of the two independent evaluations (recurrence in C, chunked WY form in
  numpy) in the forward and the backward;
* identity padding, linearity in (V, S0) and in (dO, dS_T), varlen = separate runs.

A plausible slip anywhere in the oracle (a dropped term, a wrong sign, an index
off by one, a transposed operand) breaks at least one of these.
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import chunked

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def make_problem(rng, lens, Hk=1, Hv=1, DK=8, DV=8, S0=True, dST=True, beta=None, g=None):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T, N = int(cu[-1]), len(lens)
    q = rng.standard_normal((T, Hk, DK))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((T, Hk, DK))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, Hv, DV))
    dO = rng.standard_normal((T, Hv, DV))
    gg = np.log(1.0 / (1.0 + np.exp(-rng.standard_normal((T, Hv))))) if g is None else g
    bb = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, Hv)))) if beta is None else beta
    s0 = 0.1 * rng.standard_normal((N, Hv, DV, DK)) if S0 else None
    dst = 0.1 * rng.standard_normal((N, Hv, DV, DK)) if dST else None
    return dict(cu=cu, Hk=Hk, Hv=Hv, scale=1.0 / np.sqrt(DK), q=q, k=k, v=v, g=gg, beta=bb, S0=s0, dO=dO,
                dST=dst)


def fwd(p, **kw):
    return oracle.recurrent_forward(p["cu"], p["Hk"], p["Hv"], p["scale"], p["q"], p["k"], p["v"], p["g"],
                                    p["beta"], p["S0"], **kw)


def bwd(p):
    return oracle.recurrent_backward(p["cu"], p["Hk"], p["Hv"], p["scale"], p["q"], p["k"], p["v"], p["g"],
                                     p["beta"], p["S0"], p["dO"], p["dST"])


def relmax(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


# ---------------------------------------------------------------- hand-worked example
def test_hand_worked_2x2_example():
    d = json.load(open(os.path.join(GOLDEN, "hand_2x2.json")))
    q = np.array(d["q"])[:, None, :]
    k = np.array(d["k"])[:, None, :]
    v = np.array(d["v"])[:, None, :]
    dO = np.array(d["dO"])[:, None, :]
    g = np.array(d["g"])[:, None]
    b = np.array(d["beta"])[:, None]
    cu = np.array([0, 2])
    e = d["expect"]
    o, ST, _ = oracle.recurrent_forward(cu, 1, 1, d["scale"], q, k, v, g, b)
    np.testing.assert_allclose(o[:, 0], e["o"], atol=1e-14)
    np.testing.assert_allclose(ST[0, 0], e["S_T"], atol=1e-14)
    _, _, dv, _, dbeta, _ = oracle.recurrent_backward(cu, 1, 1, d["scale"], q, k, v, g, b, None, dO, None)
    np.testing.assert_allclose(dv[:, 0], e["dv"], atol=1e-14)
    np.testing.assert_allclose(dbeta[:, 0], e["dbeta"], atol=1e-14)
    # the chunked form must reproduce the same hand values
    o2, ST2, _ = chunked.chunked_forward(cu, 1, 1, d["scale"], q, k, v, g, b)
    np.testing.assert_allclose(o2[:, 0], e["o"], atol=1e-14)
    np.testing.assert_allclose(ST2[0, 0], e["S_T"], atol=1e-14)
    r = chunked.chunked_backward(cu, 1, 1, d["scale"], q, k, v, g, b, None, dO, None)
    np.testing.assert_allclose(r[2][:, 0], e["dv"], atol=1e-14)
    np.testing.assert_allclose(r[4][:, 0], e["dbeta"], atol=1e-14)


# ---------------------------------------------------------------- finite differences
@pytest.mark.parametrize("lens,Hv,D", [([1], 1, 4), ([5], 2, 4), ([64], 1, 8), ([65], 2, 8), ([130], 1, 4),
                                       ([3, 70], 2, 4)])
def test_gradients_match_central_differences(rng, lens, Hv, D):
    p = make_problem(rng, lens, Hk=1, Hv=Hv, DK=D, DV=D)
    grads = dict(zip(["q", "k", "v", "g", "beta", "S0"], bwd(p)))

    def loss(pp):
        o, ST, _ = fwd(pp, want_chunks=False, nthreads=1)
        return float((o * pp["dO"]).sum() + (ST * pp["dST"]).sum())

    for name, gname in [("q", "q"), ("k", "k"), ("v", "v"), ("g", "g"), ("beta", "beta"), ("S0", "S0")]:
        x = p[name]
        grad = grads[gname]
        gmax = max(np.abs(grad).max(), 1e-12)
        flat = np.arange(x.size)
        picks = rng.choice(flat, size=min(12, x.size), replace=False)
        for f in picks:
            idx = np.unravel_index(f, x.shape)
            x0 = x[idx]
            eps = 1e-6 * max(1.0, abs(x0))
            x[idx] = x0 + eps
            lp = loss(p)
            x[idx] = x0 - eps
            lm = loss(p)
            x[idx] = x0
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) / gmax < 1e-6, (name, idx, fd, grad[idx])


# ---------------------------------------------------------------- beta = 0 closed form
def test_beta_zero_closed_form(rng):
    L, D = 70, 6
    p = make_problem(rng, [L], DK=D, DV=D, beta=np.zeros((L, 1)))
    c = p["scale"]
    S0 = p["S0"][0, 0]
    dST = p["dST"][0, 0]
    g = p["g"][:, 0]
    Lam = np.cumsum(g)
    q, k, v, dO = p["q"][:, 0], p["k"][:, 0], p["v"][:, 0], p["dO"][:, 0]
    o, ST, Sc = fwd(p)
    o_cf = c * np.exp(Lam)[:, None] * (q @ S0.T)
    np.testing.assert_allclose(o[:, 0], o_cf, rtol=0, atol=1e-13)
    np.testing.assert_allclose(ST[0, 0], np.exp(Lam[-1]) * S0, atol=1e-15)
    # chunk-start states: S before token 64 = e^{Lambda_63} S0
    np.testing.assert_allclose(Sc[1, 0], np.exp(Lam[63]) * S0, atol=1e-15)
    dq, dk, dv, dg, dbeta, dS0 = bwd(p)
    np.testing.assert_allclose(dq[:, 0], c * np.exp(Lam)[:, None] * (dO @ S0), atol=1e-13)
    assert np.abs(dk).max() == 0.0 and np.abs(dv).max() == 0.0
    # per-token contributions to L: c e^{Lambda_s} <do_s, S0 q_s>, plus e^{Lambda_L} <dS_T, S0>
    contrib = c * np.exp(Lam) * np.einsum("ta,ab,tb->t", dO, S0, q)
    final = np.exp(Lam[-1]) * np.sum(dST * S0)
    dg_cf = np.cumsum(contrib[::-1])[::-1] + final  # g_t enters every Lambda_s with s >= t
    np.testing.assert_allclose(dg[:, 0], dg_cf, atol=1e-12)
    dS0_cf = np.exp(Lam[-1]) * dST + c * np.einsum("t,ta,tb->ab", np.exp(Lam), dO, q)
    np.testing.assert_allclose(dS0[0, 0], dS0_cf, atol=1e-12)
    # dbeta_t = (Gbar_t k_t)^T (v_t - e^{g_t} S_{t-1} k_t)
    for t in [0, 17, 63, 64, L - 1]:
        Gbar = np.exp(Lam[-1] - Lam[t]) * dST + c * sum(
            np.exp(Lam[s] - Lam[t]) * np.outer(dO[s], q[s]) for s in range(t, L))
        Sprev = (np.exp(Lam[t - 1]) if t > 0 else 1.0) * S0
        db = (Gbar @ k[t]) @ (v[t] - np.exp(g[t]) * Sprev @ k[t])
        assert abs(db - dbeta[t, 0]) < 1e-12


# ---------------------------------------------------------------- orthonormal keys: GLA closed form
def test_orthonormal_keys_reduce_to_gated_linear_attention(rng):
    L = D = 12
    p = make_problem(rng, [L], DK=D, DV=5, S0=False, dST=False)
    Qm, _ = np.linalg.qr(rng.standard_normal((D, D)))
    p["k"] = Qm.T[:, None, :].copy()  # rows of an orthogonal matrix: k_s . k_t = delta_st
    c = p["scale"]
    q, k, v, dO = p["q"][:, 0], p["k"][:, 0], p["v"][:, 0], p["dO"][:, 0]
    b, g = p["beta"][:, 0], p["g"][:, 0]
    Lam = np.cumsum(g)
    Mts = np.tril(np.exp(Lam[:, None] - Lam[None, :]) * (q @ k.T) * b[None, :] * c)
    o, ST, _ = fwd(p)
    np.testing.assert_allclose(o[:, 0], Mts @ v, atol=1e-13)
    ST_cf = sum(np.exp(Lam[-1] - Lam[s]) * b[s] * np.outer(v[s], k[s]) for s in range(L))
    np.testing.assert_allclose(ST[0, 0], ST_cf, atol=1e-13)
    dq, dk, dv, dg, dbeta, _ = bwd(p)
    E = dO @ v.T  # E[t, s] = do_t . v_s
    np.testing.assert_allclose(dv[:, 0], Mts.T @ dO, atol=1e-13)
    Dts = np.tril(np.exp(Lam[:, None] - Lam[None, :])) * b[None, :] * c * E
    np.testing.assert_allclose(dq[:, 0], Dts @ k, atol=1e-13)
    decay = np.tril(np.exp(Lam[:, None] - Lam[None, :]))
    dbeta_cf = c * np.sum(decay * (q @ k.T) * E, axis=0)
    np.testing.assert_allclose(dbeta[:, 0], dbeta_cf, atol=1e-13)
    C = Mts * E  # C[t, s]: contribution of (t, s); g_r sits in Lambda_t - Lambda_s iff s < r <= t
    dg_cf = np.array([sum(C[t, s] for t in range(r, L) for s in range(r)) for r in range(L)])
    np.testing.assert_allclose(dg[:, 0], dg_cf, atol=1e-13)


# ---------------------------------------------------------------- exact overwrite
def test_exact_overwrite_invariant(rng):
    L, D = 150, 8
    p = make_problem(rng, [L], DK=D, DV=D, beta=np.ones((L, 1)))
    p["q"] = p["k"].copy()  # o_t = c S_t k_t = c v_t whatever the gate
    o, _, _ = fwd(p)
    np.testing.assert_allclose(o[:, 0], p["scale"] * p["v"][:, 0], atol=1e-12)
    p["g"] = np.zeros((L, 1))  # and at alpha = 1
    o, _, _ = fwd(p)
    np.testing.assert_allclose(o[:, 0], p["scale"] * p["v"][:, 0], atol=1e-12)


# ---------------------------------------------------------------- chunked vs recurrent
@pytest.mark.parametrize("lens,Hk,Hv,DK,DV,S0", [([1], 1, 1, 4, 4, True), ([63], 1, 1, 8, 8, False),
                                                 ([64], 1, 2, 8, 4, True), ([65], 2, 2, 4, 8, True),
                                                 ([130, 1, 64], 1, 2, 8, 8, True), ([200], 2, 4, 16, 8, False)])
def test_chunked_form_agrees_with_recurrence(rng, lens, Hk, Hv, DK, DV, S0):
    p = make_problem(rng, lens, Hk, Hv, DK, DV, S0=S0, dST=S0)
    o, ST, Sc = fwd(p)
    o2, ST2, Sc2 = chunked.chunked_forward(p["cu"], Hk, Hv, p["scale"], p["q"], p["k"], p["v"], p["g"],
                                           p["beta"], p["S0"])
    assert relmax(o2, o) < 1e-10 and relmax(ST2, ST) < 1e-10
    if np.abs(Sc).max() > 0:
        assert relmax(Sc2, Sc) < 1e-10
    r = bwd(p)
    r2 = chunked.chunked_backward(p["cu"], Hk, Hv, p["scale"], p["q"], p["k"], p["v"], p["g"], p["beta"],
                                  p["S0"], p["dO"], p["dST"])
    for name, a, b in zip(["dq", "dk", "dv", "dg", "dbeta", "dS0"], r2, r):
        assert relmax(a, b) < 1e-10, name


# ---------------------------------------------------------------- identity padding
def test_identity_padding(rng):
    L, P, D = 70, 30, 8
    p = make_problem(rng, [L], DK=D, DV=D)
    pad = make_problem(rng, [L + P], DK=D, DV=D)
    for key in ["q", "k", "v", "g", "beta", "dO"]:
        pad[key][:L] = p[key]
    pad["g"][L:] = 0.0
    pad["beta"][L:] = 0.0
    pad["dO"][L:] = 0.0
    pad["S0"], pad["dST"] = p["S0"], p["dST"]
    o, ST, _ = fwd(p)
    o2, ST2, _ = fwd(pad)
    np.testing.assert_allclose(o2[:L], o, atol=1e-14)
    np.testing.assert_allclose(ST2, ST, atol=1e-14)
    r, r2 = bwd(p), bwd(pad)
    for a, b in zip(r2[:5], r[:5]):
        np.testing.assert_allclose(a[:L], b, atol=1e-13)
    np.testing.assert_allclose(r2[5], r[5], atol=1e-13)
    assert np.abs(r2[1][L:]).max() == 0.0 and np.abs(r2[2][L:]).max() == 0.0  # dk, dv of padding


# ---------------------------------------------------------------- linearity
def test_linearity(rng):
    D = 8
    p1 = make_problem(rng, [90], DK=D, DV=D)
    p2 = {k_: (v_.copy() if isinstance(v_, np.ndarray) else v_) for k_, v_ in p1.items()}
    p2["v"] = rng.standard_normal(p1["v"].shape)
    p2["S0"] = 0.1 * rng.standard_normal(p1["S0"].shape)
    a, b = 0.7, -1.3
    p3 = dict(p1)
    p3["v"] = a * p1["v"] + b * p2["v"]
    p3["S0"] = a * p1["S0"] + b * p2["S0"]
    (o1, s1, _), (o2, s2, _), (o3, s3, _) = fwd(p1), fwd(p2), fwd(p3)
    np.testing.assert_allclose(o3, a * o1 + b * o2, atol=1e-12)
    np.testing.assert_allclose(s3, a * s1 + b * s2, atol=1e-12)
    # gradients are linear in (dO, dS_T)
    q2 = dict(p1)
    q2["dO"] = rng.standard_normal(p1["dO"].shape)
    q2["dST"] = 0.1 * rng.standard_normal(p1["dST"].shape)
    q3 = dict(p1)
    q3["dO"] = a * p1["dO"] + b * q2["dO"]
    q3["dST"] = a * p1["dST"] + b * q2["dST"]
    for x1, x2, x3 in zip(bwd(p1), bwd(q2), bwd(q3)):
        np.testing.assert_allclose(x3, a * x1 + b * x2, atol=1e-11)


# ---------------------------------------------------------------- varlen
def test_varlen_equals_separate_runs(rng):
    lens = [70, 1, 128, 33]
    p = make_problem(rng, lens, Hk=1, Hv=2, DK=8, DV=4)
    o, ST, Sc = fwd(p)
    r = bwd(p)
    cu = p["cu"]
    co = oracle.chunk_offsets(cu)
    for n in range(len(lens)):
        t0, t1 = cu[n], cu[n + 1]
        s = {k_: v_ for k_, v_ in p.items()}
        for key in ["q", "k", "v", "g", "beta", "dO"]:
            s[key] = p[key][t0:t1]
        s["S0"], s["dST"] = p["S0"][n:n + 1], p["dST"][n:n + 1]
        s["cu"] = np.array([0, t1 - t0])
        o1, ST1, Sc1 = fwd(s)
        assert np.array_equal(o1, o[t0:t1]) and np.array_equal(ST1[0], ST[n])
        assert np.array_equal(Sc1, Sc[co[n]:co[n + 1]])
        r1 = bwd(s)
        for a, b in zip(r1[:5], r[:5]):
            assert np.array_equal(a, b[t0:t1])
        assert np.array_equal(r1[5][0], r[5][n])


# ---------------------------------------------------------------- contract mapping
def test_reference_layouts_are_transposes():
    import torch

    from chunked_gated_delta_04_gb300.inputs import make_inputs, small_workload

    w = small_workload("t", dtype=torch.float32, T=70, Hk=1, Hv=2, DK=8, DV=4, layout="KV")
    inp = make_inputs(w)
    ref_kv = oracle.reference(inp, "KV")
    inp_vk = dict(inp)
    inp_vk["S0"] = inp["S0"].transpose(-1, -2).contiguous()
    inp_vk["dS_T"] = inp["dS_T"].transpose(-1, -2).contiguous()
    ref_vk = oracle.reference(inp_vk, "VK")
    for key in ["o", "dq", "dk", "dv", "dg", "dbeta", "h_saved"]:
        assert np.array_equal(ref_kv[key], ref_vk[key]), key
    assert np.array_equal(ref_kv["S_T"], np.swapaxes(ref_vk["S_T"], -1, -2))
    assert np.array_equal(ref_kv["dS0"], np.swapaxes(ref_vk["dS0"], -1, -2))
    assert ref_kv["h_saved"].shape == (2, 2, 8, 4)


# ---------------------------------------------------------------- fused input prologue
def _raw_inputs(rng, T=70, Hk=1, Hv=2, D=8):
    return {
        "q": 2.0 * rng.standard_normal((1, T, Hk, D)), "k": 0.5 * rng.standard_normal((1, T, Hk, D)),
        "v": rng.standard_normal((1, T, Hv, D)), "dO": rng.standard_normal((1, T, Hv, D)),
        "g": rng.standard_normal((1, T, Hv)), "beta": rng.standard_normal((1, T, Hv)),
        "S0": 0.1 * rng.standard_normal((1, Hv, D, D)), "dS_T": 0.1 * rng.standard_normal((1, Hv, D, D)),
        "cu_seqlens": None,
    }


def test_prologue_maps_closed_values():
    from oracle import prologue as pl

    np.testing.assert_allclose(pl.logsigmoid(np.array([0.0])), [-np.log(2.0)], rtol=1e-15)
    np.testing.assert_allclose(pl.sigmoid(np.array([0.0, np.log(3.0)])), [0.5, 0.75], rtol=1e-15)
    # extreme logits stay finite and take their limits
    big = np.array([-1000.0, 1000.0])
    np.testing.assert_allclose(pl.logsigmoid(big), [-1000.0, 0.0], atol=1e-300)
    np.testing.assert_allclose(pl.sigmoid(big), [0.0, 1.0], atol=1e-300)
    x_hat, s = pl.l2norm(np.array([[3.0, 4.0]]))
    np.testing.assert_allclose(x_hat, [[3.0 / np.sqrt(25 + 1e-6), 4.0 / np.sqrt(25 + 1e-6)]], rtol=1e-15)
    np.testing.assert_allclose(s, [[1.0 / np.sqrt(25 + 1e-6)]], rtol=1e-15)


def test_prologue_without_flags_is_the_operator(rng):
    from oracle import prologue as pl

    inp = _raw_inputs(rng)
    inp["g"] = pl.logsigmoid(inp["g"])
    inp["beta"] = pl.sigmoid(inp["beta"])
    a = pl.reference_with_prologue(inp, "KV", 0)
    b = oracle.reference(inp, "KV")
    for key in b:
        assert np.array_equal(a[key], b[key]), key


def test_prologue_forward_is_the_operator_on_mapped_inputs(rng):
    from oracle import prologue as pl

    raw = _raw_inputs(rng)
    mapped = dict(raw)
    mapped["q"] = raw["q"] / np.linalg.norm(raw["q"], axis=-1, keepdims=True)
    mapped["k"] = raw["k"] / np.linalg.norm(raw["k"], axis=-1, keepdims=True)
    mapped["g"] = np.log(1.0 / (1.0 + np.exp(-raw["g"])))
    mapped["beta"] = 1.0 / (1.0 + np.exp(-raw["beta"]))
    a = pl.reference_with_prologue(raw, "KV", 7, backward=False)
    b = oracle.reference(mapped, "KV", backward=False)
    for key in ["o", "S_T", "h_saved"]:
        assert relmax(a[key], b[key]) < 1e-6, key  # eps = 1e-6 in the norm only


@pytest.mark.parametrize("flags", [7, 1, 2, 4])
def test_prologue_gradients_match_central_differences(rng, flags):
    from oracle import prologue as pl

    inp = _raw_inputs(rng)
    if not flags & 2:
        inp["g"] = pl.logsigmoid(inp["g"])
    if not flags & 4:
        inp["beta"] = pl.sigmoid(inp["beta"])
    ref = pl.reference_with_prologue(inp, "KV", flags)
    grads = {"q": ref["dq"], "k": ref["dk"], "g": ref["dg"], "beta": ref["dbeta"]}

    def loss():
        r = pl.reference_with_prologue(inp, "KV", flags, backward=False, nthreads=1)
        return float((r["o"] * inp["dO"]).sum() + (r["S_T"] * inp["dS_T"]).sum())

    for name in ["q", "k", "g", "beta"]:
        x = inp[name]
        grad = grads[name]
        gmax = max(np.abs(grad).max(), 1e-12)
        for f in rng.choice(np.arange(x.size), size=10, replace=False):
            idx = np.unravel_index(f, x.shape)
            x0 = x[idx]
            h = 1e-6 * max(1.0, abs(x0))
            x[idx] = x0 + h
            lp = loss()
            x[idx] = x0 - h
            lm = loss()
            x[idx] = x0
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad[idx]) / gmax < 1e-6, (flags, name, idx, fd, grad[idx])
