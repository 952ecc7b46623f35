"""fp64 chunked (WY / UT-transform) form of the gated delta rule, forward and backward.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the CUDA product path.

This is the second, independent oracle path.  It evaluates the same operator as
``gdr_oracle.c`` (the token-by-token recurrence)

    S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = scale * S_t q_t

but the way the chunked method does (FlashQLA PR #34, Summary: "the chunked gated
delta rule"; the chunk length is 64 tokens), with numpy matmuls as the only library
primitive.  Notation, per chunk of c <= 64 tokens, with h := S^T (DK x DV, the
state at the chunk start):

  F1  gamma = in-chunk inclusive cumsum of g;  Gam[r, s] = exp(gamma_r - gamma_s) (r >= s)
  F2  A = strictly-lower( diag(beta) K K^T * Gam )
  F3  T = (I + A)^{-1}
  F4  W = T diag(beta e^gamma) K ;  U = T diag(beta) V
  F5  Vn = U - W h
      O  = scale * (diag(e^gamma) Q h + (Q K^T * Gam * M) Vn)      (M: lower incl. diagonal)
      h' = e^{gamma_C} h + (diag(e^{gamma_C - gamma}) K)^T Vn

and the reverse chunk walk of the backward (B1-B5: recompute, carry dh, chunk
gradients, WY backward, gate gradient with an in-chunk reverse cumsum).  Both the
recurrence and this file are pinned against each other and against finite
differences and closed forms in the tests.

Array layouts are those of ``oracle.recurrent_*`` (packed token-major, states as
S = [DV][DK]); see ``oracle/__init__.py``.
"""
from __future__ import annotations

import numpy as np

CHUNK = 64


def _chunk_ranges(L: int):
    for c0 in range(0, L, CHUNK):
        yield c0, min(c0 + CHUNK, L)


def _chunk_forward_terms(Kc, Vc, gc, bc):
    """F1-F4 for one chunk: gamma, Gam (masked), A, T, W, U, B_k, B_v."""
    c = Kc.shape[0]
    gamma = np.cumsum(gc)
    diff = gamma[:, None] - gamma[None, :]
    lower_incl = np.tril(np.ones((c, c), dtype=bool))
    Gam = np.zeros((c, c))
    Gam[lower_incl] = np.exp(diff[lower_incl])  # only r >= s: no overflow above the diagonal
    strict = np.tril(np.ones((c, c)), -1)
    A = strict * (bc[:, None] * (Kc @ Kc.T) * Gam)
    T = np.linalg.inv(np.eye(c) + A)
    Bk = (bc * np.exp(gamma))[:, None] * Kc
    Bv = bc[:, None] * Vc
    W = T @ Bk
    U = T @ Bv
    return gamma, Gam, A, T, W, U, Bk, Bv


def _head_forward(q, k, v, g, beta, S0, scale):
    """One (sequence, v-head): returns o [L,DV], S_T [DV,DK], chunk-start states [n,DV,DK]."""
    L, DK = k.shape
    DV = v.shape[1]
    h = np.zeros((DK, DV)) if S0 is None else S0.T.copy()
    o = np.zeros((L, DV))
    starts = []
    for c0, c1 in _chunk_ranges(L):
        Qc, Kc, Vc = q[c0:c1], k[c0:c1], v[c0:c1]
        gamma, Gam, A, T, W, U, Bk, Bv = _chunk_forward_terms(Kc, Vc, g[c0:c1], beta[c0:c1])
        starts.append(h.T.copy())
        Vn = U - W @ h
        P = (Qc @ Kc.T) * Gam  # Gam is already zero above the diagonal (mask M)
        o[c0:c1] = scale * (np.exp(gamma)[:, None] * (Qc @ h) + P @ Vn)
        gC = gamma[-1]
        h = np.exp(gC) * h + (np.exp(gC - gamma)[:, None] * Kc).T @ Vn
    states = np.stack(starts) if starts else np.zeros((0, DV, DK))
    return o, h.T.copy(), states


def _head_backward(q, k, v, g, beta, S0, dO, dST, scale):
    """One (sequence, v-head) reverse chunk walk.  Returns dq, dk, dv, dg, dbeta, dS0."""
    L, DK = k.shape
    DV = v.shape[1]
    ranges = list(_chunk_ranges(L))
    # B1: chunk-start states from a forward sweep (what the forward saves)
    h = np.zeros((DK, DV)) if S0 is None else S0.T.copy()
    hs = []
    for c0, c1 in ranges:
        gamma, Gam, A, T, W, U, Bk, Bv = _chunk_forward_terms(k[c0:c1], v[c0:c1], g[c0:c1], beta[c0:c1])
        hs.append(h.copy())
        Vn = U - W @ h
        gC = gamma[-1]
        h = np.exp(gC) * h + (np.exp(gC - gamma)[:, None] * k[c0:c1]).T @ Vn

    dq = np.zeros((L, DK))
    dk = np.zeros((L, DK))
    dv = np.zeros((L, DV))
    dg = np.zeros(L)
    dbeta = np.zeros(L)
    dh_next = np.zeros((DK, DV)) if dST is None else dST.T.copy()  # dL/dh at the chunk end
    for ci in range(len(ranges) - 1, -1, -1):
        c0, c1 = ranges[ci]
        Qc, Kc, Vc, dOc = q[c0:c1], k[c0:c1], v[c0:c1], dO[c0:c1]
        bc = beta[c0:c1]
        h = hs[ci]
        gamma, Gam, A, T, W, U, Bk, Bv = _chunk_forward_terms(Kc, Vc, g[c0:c1], bc)
        eg = np.exp(gamma)
        gC = gamma[-1]
        dec = np.exp(gC - gamma)  # e^{gamma_C - gamma_r}
        Vn = U - W @ h
        P = (Qc @ Kc.T) * Gam
        Kt = dec[:, None] * Kc  # K tilde
        Qh = eg[:, None] * Qc  # Q hat

        # B2: dVn and the state gradient at the chunk start
        dVn = scale * P.T @ dOc + Kt @ dh_next
        dh = np.exp(gC) * dh_next + scale * Qh.T @ dOc - W.T @ dVn

        # B3: in-chunk gradients of the output and state-update terms
        dP = scale * (dOc @ Vn.T) * Gam  # masked: gradient w.r.t. (Q K^T) entries
        dQc = scale * eg[:, None] * (dOc @ h.T) + dP @ Kc
        dKc = dP.T @ Qc + dec[:, None] * (Vn @ dh_next.T)
        dW = -dVn @ h.T
        dU = dVn

        # B4: WY backward through W = T B_k, U = T B_v, T = (I + A)^{-1}
        dT = dW @ Bk.T + dU @ Bv.T
        dBk = T.T @ dW
        dBv = T.T @ dU
        dA = -(T.T @ dT @ T.T)
        dA = np.tril(dA, -1)
        KK = Kc @ Kc.T
        dAG = dA * Gam
        dVc = bc[:, None] * dBv
        dKc += (bc * eg)[:, None] * dBk
        dKc += bc[:, None] * (dAG @ Kc) + dAG.T @ (bc[:, None] * Kc)
        dbc = eg * np.sum(dBk * Kc, axis=1) + np.sum(dBv * Vc, axis=1) + np.sum(dAG * KK, axis=1)

        # B5: gradient w.r.t. the in-chunk cumsum gamma, then dg = reverse cumsum
        dgam = np.sum(dBk * Bk, axis=1)
        dAA = dA * A
        dgam += dAA.sum(axis=1) - dAA.sum(axis=0)
        dPP = dP * (Qc @ Kc.T)  # = (dL/dP) * P, since dP already carries Gam
        dgam += dPP.sum(axis=1) - dPP.sum(axis=0)
        dgam += scale * eg * np.sum(dOc * (Qc @ h), axis=1)
        kdv = np.sum((Kc @ dh_next) * Vn, axis=1)  # k_r^T dh' vn_r
        dgam -= dec * kdv
        dgam[-1] += np.exp(gC) * np.sum(dh_next * h) + np.sum(dec * kdv)
        dgc = np.cumsum(dgam[::-1])[::-1]

        dq[c0:c1] = dQc
        dk[c0:c1] = dKc
        dv[c0:c1] = dVc
        dg[c0:c1] = dgc
        dbeta[c0:c1] = dbc
        dh_next = dh
    return dq, dk, dv, dg, dbeta, dh_next.T.copy()


def chunked_forward(cu_seqlens, Hk, Hv, scale, q, k, v, g, beta, S0=None):
    """Chunked forward over a packed batch.  Returns (o, S_T, S_chunks)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    G = Hv // Hk
    DK, DV = q.shape[2], v.shape[2]
    o = np.zeros((q.shape[0], Hv, DV))
    S_T = np.zeros((N, Hv, DV, DK))
    chunks = []
    for n in range(N):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        nc = (t1 - t0 + CHUNK - 1) // CHUNK
        st = np.zeros((nc, Hv, DV, DK))
        for j in range(Hv):
            i = j // G
            s0 = None if S0 is None else S0[n, j]
            oo, sT, states = _head_forward(q[t0:t1, i], k[t0:t1, i], v[t0:t1, j], g[t0:t1, j],
                                           beta[t0:t1, j], s0, scale)
            o[t0:t1, j] = oo
            S_T[n, j] = sT
            st[:, j] = states
        chunks.append(st)
    S_chunks = np.concatenate(chunks, axis=0) if chunks else np.zeros((0, Hv, DV, DK))
    return o, S_T, S_chunks


def chunked_backward(cu_seqlens, Hk, Hv, scale, q, k, v, g, beta, S0, dO, dS_T):
    """Chunked backward over a packed batch.  Returns (dq, dk, dv, dg, dbeta, dS0)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    G = Hv // Hk
    DK, DV = q.shape[2], v.shape[2]
    dq = np.zeros_like(q, dtype=np.float64)
    dk = np.zeros_like(k, dtype=np.float64)
    dv = np.zeros((v.shape[0], Hv, DV))
    dg = np.zeros((g.shape[0], Hv))
    dbeta = np.zeros((g.shape[0], Hv))
    dS0 = np.zeros((N, Hv, DV, DK))
    for n in range(N):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for j in range(Hv):
            i = j // G
            s0 = None if S0 is None else S0[n, j]
            dst = None if dS_T is None else dS_T[n, j]
            r = _head_backward(q[t0:t1, i], k[t0:t1, i], v[t0:t1, j], g[t0:t1, j], beta[t0:t1, j],
                               s0, dO[t0:t1, j], dst, scale)
            dq[t0:t1, i] += r[0]
            dk[t0:t1, i] += r[1]
            dv[t0:t1, j] = r[2]
            dg[t0:t1, j] = r[3]
            dbeta[t0:t1, j] = r[4]
            dS0[n, j] = r[5]
    return dq, dk, dv, dg, dbeta, dS0
