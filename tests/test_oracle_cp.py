"""Pins for the segment-scan (intra-card context parallel) oracle, CPU only.

The segment-scan evaluation must reproduce the token recurrence (C) and the chunked form
exactly (fp64, up to rounding order) for any cut of a sequence into segments; its per-segment
maps must compose like the chunks they cover; and with beta = 0 they reduce to the closed
form of a pure decay.
"""
import numpy as np
import pytest

from oracle import chunked, context_parallel as cp

from test_oracle_pins import bwd, fwd, make_problem, relmax


@pytest.mark.parametrize("lens,Hk,Hv,D,S0,n_seg", [
    ([200], 1, 1, 8, True, 1),
    ([200], 1, 1, 8, True, 2),
    ([330], 1, 2, 8, True, 3),            # ragged last chunk, two v-heads per q/k head
    ([0, 1, 64, 65, 200], 1, 2, 8, True, 2),  # empty, one token, one chunk, ragged tail
    ([640], 2, 2, 16, False, 7),          # ten chunks in seven segments of one or two chunks
    ([129], 1, 1, 4, True, 5),            # more segments asked for than there are chunks
])
def test_segment_scan_matches_recurrence_and_chunked_form(rng, lens, Hk, Hv, D, S0, n_seg):
    p = make_problem(rng, lens, Hk, Hv, D, D, S0=S0, dST=S0)
    args = (p["cu"], Hk, Hv, p["scale"], p["q"], p["k"], p["v"], p["g"], p["beta"])
    o, ST, Sc = fwd(p)
    o2, ST2, Sc2 = cp.cp_forward(*args, p["S0"], n_segments=n_seg)
    o3, ST3, Sc3 = chunked.chunked_forward(*args, p["S0"])
    assert relmax(o2, o) < 1e-10 and relmax(ST2, ST) < 1e-10
    assert relmax(o2, o3) < 1e-12
    if np.abs(Sc3).max() > 0:  # the saved chunk-start states (all zero when S0 = 0 and L <= 64)
        assert relmax(Sc2, Sc3) < 1e-12
    r = bwd(p)
    r2 = cp.cp_backward(*args, p["S0"], p["dO"], p["dST"], n_segments=n_seg)
    for name, a, b in zip(["dq", "dk", "dv", "dg", "dbeta", "dS0"], r2, r):
        assert relmax(a, b) < 1e-10, name


def test_segment_maps_compose(rng):
    # the map of chunks [0, 5) is the map of [2, 5) applied after the map of [0, 2); the same
    # for the gradient maps in reverse: this is what lets the segments run side by side
    p = make_problem(rng, [300], DK=8, DV=8)
    k, v, g, b = p["k"][:, 0], p["v"][:, 0], p["g"][:, 0], p["beta"][:, 0]
    q, dO = p["q"][:, 0], p["dO"][:, 0]
    Pa, Ra = cp.segment_map(k, v, g, b, 0, 2)
    Pb, Rb = cp.segment_map(k, v, g, b, 2, 5)
    P, R = cp.segment_map(k, v, g, b, 0, 5)
    assert relmax(Pb @ Pa, P) < 1e-13 and relmax(Pb @ Ra + Rb, R) < 1e-13
    Ea = cp.segment_grad_map(q, k, v, g, b, dO, p["scale"], 0, 2)
    Eb = cp.segment_grad_map(q, k, v, g, b, dO, p["scale"], 2, 5)
    E = cp.segment_grad_map(q, k, v, g, b, dO, p["scale"], 0, 5)
    assert relmax(Pa.T @ Eb + Ea, E) < 1e-13


def test_pure_decay_maps(rng):
    # beta = 0: no writes, so Phi = e^{sum g} I, R = 0, and the gradient map is the decayed
    # sum of the output terms, E = scale sum_t e^{Lambda_t} q_t dO_t^T (Lambda from the
    # segment start, t included)
    L, D = 150, 8
    p = make_problem(rng, [L], DK=D, DV=D, beta=np.zeros((L, 1)))
    k, v, g, b = p["k"][:, 0], p["v"][:, 0], p["g"][:, 0], p["beta"][:, 0]
    q, dO = p["q"][:, 0], p["dO"][:, 0]
    Phi, R = cp.segment_map(k, v, g, b, 1, 3)  # tokens 64 .. 149
    lam = np.cumsum(g[64:150])
    assert relmax(Phi, np.exp(lam[-1]) * np.eye(D)) < 1e-13
    assert np.abs(R).max() == 0.0
    E = cp.segment_grad_map(q, k, v, g, b, dO, p["scale"], 1, 3)
    E_ref = p["scale"] * (np.exp(lam)[:, None] * q[64:150]).T @ dO[64:150]
    assert relmax(E, E_ref) < 1e-13


def test_split_chunks():
    assert cp.split_chunks(10, 3) == [(0, 4), (4, 7), (7, 10)]
    assert cp.split_chunks(2, 5) == [(0, 1), (1, 2)]
    assert cp.split_chunks(0, 4) == []
    assert cp.split_chunks(7, 1) == [(0, 7)]
