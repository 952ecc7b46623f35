"""fp64 segment-scan (intra-card context parallel) evaluation of the gated delta rule.

TEST INFRASTRUCTURE ONLY: imported by the tests, never by the CUDA product path.

FlashQLA PR #34 ("Current status") lists intra-card context parallelism (CP) among the
features of the chunked gated delta rule but does not spell the scheme out.  The reading
taken here is the plainest one the chunked form supports: a sequence is cut at chunk
boundaries into segments that are processed side by side, and the sequential dependence
between them is carried by an exact affine map per segment.

Forward.  With h := S^T (DK x DV) and the chunk factors of ``oracle/chunked.py``
(gamma, W, U; K~ = diag(e^{gamma_C - gamma}) K), one chunk updates

    h' = e^{gamma_C} h + K~^T (U - W h) = A_c h + b_c,
    A_c = e^{gamma_C} I - K~^T W   (DK x DK),   b_c = K~^T U   (DK x DV),

so a segment of chunks c1..cm maps its start state to its end state by
h_end = Phi h_start + R with Phi = A_cm ... A_c1 and R the end state reached from h = 0.
Step 1 computes (Phi_s, R_s) of every segment independently; step 2 scans the segments in
order, h_start(s + 1) = Phi_s h_start(s) + R_s from h_start(0) = S0^T; step 3 evaluates
every segment again from its true start state (outputs, saved chunk states).

Backward.  The reverse chunk walk of the backward is affine in the state gradient too:

    dh = e^{gamma_C} dh' + scale Q~^T dO - W^T dVn,  dVn = scale P^T dO + K~ dh'
       = A_c^T dh' + e_c,   e_c = scale (Q~ - P W)^T dO,   Q~ = diag(e^gamma) Q,

so a segment maps the gradient at its end to the gradient at its start by
dh_start = Phi_s^T dh_end + E_s, E_s being the walk from dh_end = 0.  Step 1' computes E_s
per segment (Phi_s is shared with the forward), step 2' scans from the last segment,
dh_end(last) = dS_T^T and dh_end(s - 1) = Phi_s^T dh_end(s) + E_s, and step 3' runs every
segment's full backward with its true start state and end gradient.

Array layouts are those of ``oracle.recurrent_*`` (packed token-major, states S = [DV][DK]).
"""
from __future__ import annotations

import numpy as np

from .chunked import CHUNK, _chunk_forward_terms, _head_backward, _head_forward


def split_chunks(n_chunks: int, n_segments: int):
    """Chunk index ranges [a, b) of at most n_segments non-empty segments, sizes within one."""
    n_seg = max(1, min(n_segments, n_chunks))
    if n_chunks == 0:
        return []
    base, extra = divmod(n_chunks, n_seg)
    out, a = [], 0
    for s in range(n_seg):
        b = a + base + (1 if s < extra else 0)
        out.append((a, b))
        a = b
    return out


def chunk_affine(Kc, Vc, gc, bc):
    """(A_c, b_c) of one chunk: h' = A_c h + b_c."""
    gamma, Gam, A, T, W, U, Bk, Bv = _chunk_forward_terms(Kc, Vc, gc, bc)
    gC = gamma[-1]
    Kt = np.exp(gC - gamma)[:, None] * Kc
    return np.exp(gC) * np.eye(Kc.shape[1]) - Kt.T @ W, Kt.T @ U


def chunk_grad_affine(Qc, Kc, Vc, gc, bc, dOc, scale):
    """e_c of one chunk: dh = A_c^T dh' + e_c."""
    gamma, Gam, A, T, W, U, Bk, Bv = _chunk_forward_terms(Kc, Vc, gc, bc)
    P = (Qc @ Kc.T) * Gam
    return scale * (np.exp(gamma)[:, None] * Qc - P @ W).T @ dOc


def segment_map(k, v, g, beta, c_lo, c_hi):
    """(Phi, R) of chunks c_lo..c_hi-1 of one (sequence, v-head): h_end = Phi h_start + R."""
    L, DK = k.shape
    DV = v.shape[1]
    Phi, R = np.eye(DK), np.zeros((DK, DV))
    for c in range(c_lo, c_hi):
        t0, t1 = c * CHUNK, min((c + 1) * CHUNK, L)
        Ac, bcv = chunk_affine(k[t0:t1], v[t0:t1], g[t0:t1], beta[t0:t1])
        Phi, R = Ac @ Phi, Ac @ R + bcv
    return Phi, R


def segment_grad_map(q, k, v, g, beta, dO, scale, c_lo, c_hi):
    """E of chunks c_lo..c_hi-1: the state gradient at the segment start from a zero end gradient."""
    L, DK = k.shape
    DV = v.shape[1]
    E = np.zeros((DK, DV))
    for c in range(c_hi - 1, c_lo - 1, -1):
        t0, t1 = c * CHUNK, min((c + 1) * CHUNK, L)
        Ac, _ = chunk_affine(k[t0:t1], v[t0:t1], g[t0:t1], beta[t0:t1])
        E = Ac.T @ E + chunk_grad_affine(q[t0:t1], k[t0:t1], v[t0:t1], g[t0:t1], beta[t0:t1], dO[t0:t1], scale)
    return E


def _segment_starts(k, v, g, beta, S0, segs):
    """Steps 1-2: the true start state h of every segment (scan over the segments' maps)."""
    DK, DV = k.shape[1], v.shape[1]
    maps = [segment_map(k, v, g, beta, a, b) for a, b in segs]  # independent per segment
    h = np.zeros((DK, DV)) if S0 is None else S0.T.copy()
    starts = []
    for Phi, R in maps:
        starts.append(h)
        h = Phi @ h + R
    return starts, maps, h


def _head_cp_forward(q, k, v, g, beta, S0, scale, n_segments):
    L, DK = k.shape
    DV = v.shape[1]
    segs = split_chunks((L + CHUNK - 1) // CHUNK, n_segments)
    starts, maps, h_end = _segment_starts(k, v, g, beta, S0, segs)
    o = np.zeros((L, DV))
    states = []
    for (a, b), h0 in zip(segs, starts):  # step 3: each segment from its true start state
        t0, t1 = a * CHUNK, min(b * CHUNK, L)
        oo, sT, st = _head_forward(q[t0:t1], k[t0:t1], v[t0:t1], g[t0:t1], beta[t0:t1], h0.T, scale)
        o[t0:t1] = oo
        states.append(st)
    S_T = h_end.T.copy() if segs else (np.zeros((DV, DK)) if S0 is None else S0.copy())
    return o, S_T, (np.concatenate(states) if states else np.zeros((0, DV, DK)))


def _head_cp_backward(q, k, v, g, beta, S0, dO, dST, scale, n_segments):
    L, DK = k.shape
    DV = v.shape[1]
    segs = split_chunks((L + CHUNK - 1) // CHUNK, n_segments)
    starts, maps, _ = _segment_starts(k, v, g, beta, S0, segs)
    Es = [segment_grad_map(q, k, v, g, beta, dO, scale, a, b) for a, b in segs]  # step 1'
    dh = np.zeros((DK, DV)) if dST is None else dST.T.copy()
    ends = [None] * len(segs)
    for s in range(len(segs) - 1, -1, -1):  # step 2': scan from the last segment
        ends[s] = dh
        dh = maps[s][0].T @ dh + Es[s]
    dq, dk = np.zeros((L, DK)), np.zeros((L, DK))
    dv, dg, dbeta = np.zeros((L, DV)), np.zeros(L), np.zeros(L)
    for (a, b), h0, dh1 in zip(segs, starts, ends):  # step 3': each segment's own backward
        t0, t1 = a * CHUNK, min(b * CHUNK, L)
        r = _head_backward(q[t0:t1], k[t0:t1], v[t0:t1], g[t0:t1], beta[t0:t1], h0.T, dO[t0:t1], dh1.T, scale)
        dq[t0:t1], dk[t0:t1], dv[t0:t1], dg[t0:t1], dbeta[t0:t1] = r[:5]
    dS0 = dh.T.copy() if segs else (np.zeros((DV, DK)) if dST is None else dST.copy())
    return dq, dk, dv, dg, dbeta, dS0


def cp_forward(cu_seqlens, Hk, Hv, scale, q, k, v, g, beta, S0=None, n_segments=2):
    """Segment-scan forward over a packed batch.  Returns (o, S_T, S_chunks) like chunked_forward."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N, G = len(cu) - 1, Hv // Hk
    DK, DV = q.shape[2], v.shape[2]
    o = np.zeros((q.shape[0], Hv, DV))
    S_T = np.zeros((N, Hv, DV, DK))
    chunks = []
    for n in range(N):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        st = np.zeros(((t1 - t0 + CHUNK - 1) // CHUNK, Hv, DV, DK))
        for j in range(Hv):
            i = j // G
            s0 = None if S0 is None else S0[n, j]
            oo, sT, states = _head_cp_forward(q[t0:t1, i], k[t0:t1, i], v[t0:t1, j], g[t0:t1, j],
                                              beta[t0:t1, j], s0, scale, n_segments)
            o[t0:t1, j], S_T[n, j], st[:, j] = oo, sT, states
        chunks.append(st)
    return o, S_T, (np.concatenate(chunks, axis=0) if chunks else np.zeros((0, Hv, DV, DK)))


def cp_backward(cu_seqlens, Hk, Hv, scale, q, k, v, g, beta, S0, dO, dS_T, n_segments=2):
    """Segment-scan backward over a packed batch.  Returns (dq, dk, dv, dg, dbeta, dS0)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N, G = len(cu) - 1, Hv // Hk
    DK, DV = q.shape[2], v.shape[2]
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros((v.shape[0], Hv, DV))
    dg = np.zeros((g.shape[0], Hv))
    dbeta = np.zeros((g.shape[0], Hv))
    dS0 = np.zeros((N, Hv, DV, DK))
    for n in range(N):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for j in range(Hv):
            i = j // G
            r = _head_cp_backward(q[t0:t1, i], k[t0:t1, i], v[t0:t1, j], g[t0:t1, j], beta[t0:t1, j],
                                  None if S0 is None else S0[n, j], dO[t0:t1, j],
                                  None if dS_T is None else dS_T[n, j], scale, n_segments)
            dq[t0:t1, i] += r[0]
            dk[t0:t1, i] += r[1]
            dv[t0:t1, j], dg[t0:t1, j], dbeta[t0:t1, j], dS0[n, j] = r[2], r[3], r[4], r[5]
    return dq, dk, dv, dg, dbeta, dS0
