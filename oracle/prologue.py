"""Oracle of the fused input prologue (plain fp64 numpy).  TEST INFRASTRUCTURE ONLY:
like the rest of ``oracle/``, only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may use it.

The operator's callers usually prepare its inputs the same way: q and k are
L2-normalised per token and head, the log decay is g = logsigmoid(a) of a raw gate
logit a, and beta = sigmoid(b) of a raw logit b (the pages list the gated delta rule's
inputs as given; the benchmark workloads apply these maps outside the operator).  With
the prologue the operator takes the raw q, k, a, b and returns gradients with respect
to them.  Definitions (the plainest reading; eps guards a zero vector):

    q_hat = q * s_q,  s_q = (sum_i q_i^2 + eps)^(-1/2),  eps = 1e-6   (same for k)
    g     = logsigmoid(a) = min(a, 0) - log(1 + exp(-|a|))
    beta  = sigmoid(b)    = 1 / (1 + exp(-b))

and their backward by the chain rule:

    dq    = s_q (dq_hat - q_hat <q_hat, dq_hat>)
    da    = dg * sigmoid(-a)
    db    = dbeta * beta (1 - beta)

Parity pinned in tests/test_oracle_pins.py: central finite differences of the composed
loss with respect to the raw inputs, closed values of the three maps, and the identity
when no prologue bit is set.
"""
from __future__ import annotations

import numpy as np

from . import reference

EPS = 1e-6
QK_L2NORM = 1
G_LOGSIGMOID = 2
BETA_SIGMOID = 4


def _np(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def l2norm(x):
    """Returns (x * s, s) with s = (sum over the last axis of x^2 + EPS)^(-1/2)."""
    s = 1.0 / np.sqrt((x * x).sum(-1, keepdims=True) + EPS)
    return x * s, s


def l2norm_backward(x_hat, s, dx_hat):
    return s * (dx_hat - x_hat * (x_hat * dx_hat).sum(-1, keepdims=True))


def logsigmoid(a):
    return np.minimum(a, 0.0) - np.log1p(np.exp(-np.abs(a)))


def sigmoid(b):
    e = np.exp(-np.abs(b))
    return np.where(b >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def reference_with_prologue(inp: dict, layout: str, flags: int, backward: bool = True, nthreads=None) -> dict:
    """``oracle.reference`` on raw inputs: ``inp["q"], inp["k"]`` are the raw q, k when
    QK_L2NORM is set, ``inp["g"]`` the raw gate logit a when G_LOGSIGMOID is set and
    ``inp["beta"]`` the raw logit b when BETA_SIGMOID is set.  Gradients are with
    respect to those raw tensors; every other output is the operator's."""
    eff = dict(inp)
    q, k, a, b = (_np(inp[n]) for n in ("q", "k", "g", "beta"))
    if flags & QK_L2NORM:
        q_hat, s_q = l2norm(q)
        k_hat, s_k = l2norm(k)
        eff["q"], eff["k"] = q_hat, k_hat
    if flags & G_LOGSIGMOID:
        eff["g"] = logsigmoid(a)
    if flags & BETA_SIGMOID:
        beta = sigmoid(b)
        eff["beta"] = beta
    out = reference(eff, layout, backward=backward, nthreads=nthreads)
    if backward:
        if flags & QK_L2NORM:
            out["dq"] = l2norm_backward(q_hat, s_q, out["dq"])
            out["dk"] = l2norm_backward(k_hat, s_k, out["dk"])
        if flags & G_LOGSIGMOID:
            out["dg"] = out["dg"] * sigmoid(-a)
        if flags & BETA_SIGMOID:
            out["dbeta"] = out["dbeta"] * beta * (1.0 - beta)
    return out
