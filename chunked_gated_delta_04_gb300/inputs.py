"""Seeded synthetic inputs for the gated delta rule (shared by the tests, the bench
and the oracle's callers; holds none of the operator's arithmetic).

Recipe (all draws fp32 from one ``torch.Generator`` seeded with ``seed``, on the CPU,
in this order): sequence lengths (varlen only), q, k, v, dO, g-logits, beta-logits,
S0, dS_T.  Then q and k are L2-normalised per token, g = logsigmoid(x + g_shift),
beta = sigmoid(x), and q, k, v, dO, beta are cast to the compute dtype.  g, S0 and
dS_T stay fp32; S0 and dS_T are 0.1 * N(0, 1) drawn directly in the storage layout
([N, Hv, DK, DV] for "KV", [N, Hv, DV, DK] for "VK").  With ``raw=True`` (inputs of the
operator's fused prologue) the same draws are returned without the maps: q and k not
normalised, g = the gate logit x + g_shift, beta = the beta logit (cast to the dtype).

The five named workloads are the chunked gated delta rule shapes of the benchmark
(chunk 64):

  tiny_fp32     fp32, B=1, H=1, T=128, D=64, no initial/final state
  b2_t4096      bf16, B=2, T=4096, H=16, D=128, "KV" layout, S0 and dS_T given
  varlen8       bf16, 8 sequences of U{256..8192} tokens packed by cu_seqlens, H=16, D=128
  long_t65536   bf16, B=1, T=65536, H=16, D=128, "VK" layout, g = logsigmoid(N(2, 1))
  gva_b4_t8192  bf16, B=4, T=8192, Hk=16, Hv=32, D=128, no initial/final state

and two smaller cases with the same kernel choices, sized for profiler captures:
long_t16384 (B=1, T=16384, otherwise long_t65536) and gva_b2_t4096 (B=2, T=4096, otherwise
gva_b4_t8192).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch


@dataclass
class Workload:
    name: str
    dtype: torch.dtype
    B: int
    T: int
    Hk: int
    Hv: int
    DK: int
    DV: int
    layout: str = "KV"
    with_S0: bool = True
    with_dST: bool = True
    g_shift: float = 0.0
    varlen: Optional[tuple] = None  # (num_seqs, lo, hi): lengths ~ U{lo..hi}
    seqlens: Optional[list] = field(default=None)  # explicit lengths (varlen)
    seed: int = 0


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", torch.float32, 1, 128, 1, 1, 64, 64, "KV", False, False),
    "b2_t4096": Workload("b2_t4096", torch.bfloat16, 2, 4096, 16, 16, 128, 128, "KV", True, True),
    "varlen8": Workload("varlen8", torch.bfloat16, 1, 0, 16, 16, 128, 128, "KV", True, True,
                        varlen=(8, 256, 8192)),
    "long_t65536": Workload("long_t65536", torch.bfloat16, 1, 65536, 16, 16, 128, 128, "VK", True, True,
                            g_shift=2.0),
    "gva_b4_t8192": Workload("gva_b4_t8192", torch.bfloat16, 4, 8192, 16, 32, 128, 128, "KV", False, False),
    # smaller cases of the same kernels' launch configurations, for profiler captures that must
    # stay within a few GB of device memory
    "long_t16384": Workload("long_t16384", torch.bfloat16, 1, 16384, 16, 16, 128, 128, "VK", True, True,
                            g_shift=2.0),
    "gva_b2_t4096": Workload("gva_b2_t4096", torch.bfloat16, 2, 4096, 16, 32, 128, 128, "KV", False, False),
    # the long-sequence workload with 2 heads (8 chunk chains at 4 DV slices): the case intra-card
    # context parallelism is for, where the plain chains leave most SMs idle
    "long_h2_t65536": Workload("long_h2_t65536", torch.bfloat16, 1, 65536, 2, 2, 128, 128, "VK", True, True,
                               g_shift=2.0),
}


def make_inputs(w: Workload, raw: bool = False) -> dict:
    """Generate the C-ABI input tensors (CPU) for workload ``w`` (``raw``: see the module doc).

    Returns q, k [B,T,Hk,DK]; v, dO [B,T,Hv,DV] (compute dtype); g [B,T,Hv] fp32;
    beta [B,T,Hv] (compute dtype); S0, dS_T fp32 or None; cu_seqlens int32 [N+1] or None;
    plus "layout", "num_seqs" and "seqlens".
    """
    gen = torch.Generator().manual_seed(w.seed)
    if w.varlen is not None or w.seqlens is not None:
        if w.seqlens is not None:
            lens = [int(x) for x in w.seqlens]
        else:
            n, lo, hi = w.varlen
            lens = torch.randint(lo, hi + 1, (n,), generator=gen).tolist()
        B, T = 1, int(sum(lens))
        cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
        N = len(lens)
    else:
        B, T = w.B, w.T
        lens = [T] * B
        cu = None
        N = B
    f32 = torch.float32
    q = torch.randn(B, T, w.Hk, w.DK, generator=gen, dtype=f32)
    k = torch.randn(B, T, w.Hk, w.DK, generator=gen, dtype=f32)
    v = torch.randn(B, T, w.Hv, w.DV, generator=gen, dtype=f32)
    dO = torch.randn(B, T, w.Hv, w.DV, generator=gen, dtype=f32)
    g_logit = torch.randn(B, T, w.Hv, generator=gen, dtype=f32)
    b_logit = torch.randn(B, T, w.Hv, generator=gen, dtype=f32)
    sshape = (N, w.Hv, w.DK, w.DV) if w.layout == "KV" else (N, w.Hv, w.DV, w.DK)
    S0 = 0.1 * torch.randn(*sshape, generator=gen, dtype=f32) if w.with_S0 else None
    dST = 0.1 * torch.randn(*sshape, generator=gen, dtype=f32) if w.with_dST else None
    if raw:
        g, beta = g_logit + w.g_shift, b_logit
    else:
        q = torch.nn.functional.normalize(q, dim=-1)
        k = torch.nn.functional.normalize(k, dim=-1)
        g = torch.nn.functional.logsigmoid(g_logit + w.g_shift)
        beta = torch.sigmoid(b_logit)
    dt = w.dtype
    return {
        "q": q.to(dt).contiguous(), "k": k.to(dt).contiguous(), "v": v.to(dt).contiguous(),
        "dO": dO.to(dt).contiguous(), "g": g.contiguous(), "beta": beta.to(dt).contiguous(),
        "S0": S0, "dS_T": dST, "cu_seqlens": cu, "layout": w.layout, "num_seqs": N, "seqlens": lens,
    }


def small_workload(name: str, dtype=torch.bfloat16, B=1, T=130, Hk=1, Hv=1, DK=128, DV=128, layout="KV",
                   with_S0=True, with_dST=True, seqlens=None, g_shift=0.0, seed=0) -> Workload:
    """A custom (usually small) workload with the same value distributions."""
    return Workload(name, dtype, B, T, Hk, Hv, DK, DV, layout, with_S0, with_dST, g_shift, None,
                    seqlens, seed)
