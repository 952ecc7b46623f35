"""The benchmark's work model (host logic, no GPU): the algorithmic flops and compulsory bytes
behind the reported roofline fractions, pinned to values worked out by hand for three of the
benchmark shapes, and the staleness rule of the stored ncu traffic figures.

Hand values (chunk C = 64, D = 128, bf16 operands, fp32 g, states and saved chunk states):
per token-head the chunked method's GEMMs are 181.6 kFLOP forward and 476.5 kFLOP backward
(dense C x C products, the unit-triangular inverse as C^3/3) when every chunk is full and each
q/k head serves one v-head; the forward moves q, k, v, o (256 B each per token-head), g (4 B),
beta (2 B) and one fp32 128 x 128 saved state per chunk (1024 B per token-head), plus S0 and
S_T once per sequence and head; the backward moves q, k, v, dO, dq, dk, dv, g, dg, beta, dbeta,
the saved states, dS_T and dS0.  S_T and dS0 are counted whenever they are written (the
benchmark asks for both, with or without S0 and dS_T); S0 and dS_T only when given.
"""
import hashlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _model(name):
    import bench
    from chunked_gated_delta_04_gb300.inputs import WORKLOADS

    w = WORKLOADS[name]
    inp = {"seqlens": [w.T] * w.B, "num_seqs": w.B, "S0": object() if w.with_S0 else None,
           "dS_T": object() if w.with_dST else None}
    return bench.work_model(inp, w), w


@pytest.mark.parametrize(
    "name, gflop_fwd, gflop_bwd, mb_fwd, mb_bwd",
    [
        # B=2, T=4096, Hk=Hv=16, S0 and dS_T given: 131072 token-heads
        ("b2_t4096", 23.80, 62.46, 273.4, 374.9),
        # B=1, T=65536, H=16, S0 and dS_T given: 1048576 token-heads
        ("long_t65536", 190.41, 499.65, 2155.9, 2967.5),
        # B=4, T=8192, Hk=16, Hv=32 (two v-heads per q/k head: the q/k products are shared and
        # dq, dk counted once per q/k head), no S0 or dS_T
        ("gva_b4_t8192", 173.23, 482.47, 1893.7, 2436.9),
    ],
)
def test_work_model_matches_hand_values(name, gflop_fwd, gflop_bwd, mb_fwd, mb_bwd):
    m, w = _model(name)
    assert m["flops_fwd"] / 1e9 == pytest.approx(gflop_fwd, abs=0.06)
    assert m["flops_bwd"] / 1e9 == pytest.approx(gflop_bwd, abs=0.06)
    assert m["bytes_fwd"] / 1e6 == pytest.approx(mb_fwd, abs=0.06)
    assert m["bytes_bwd"] / 1e6 == pytest.approx(mb_bwd, abs=0.06)


def test_per_token_head_figures():
    # full chunks, one v-head per q/k head: the per token-head constants of the module doc
    m, w = _model("b2_t4096")
    th = w.B * w.T * w.Hv
    assert m["flops_fwd"] / th == pytest.approx(181.6e3, rel=2e-4)
    assert m["flops_bwd"] / th == pytest.approx(476.5e3, rel=2e-4)
    per_seq_states = w.B * w.Hv * 128 * 128 * 4
    assert m["bytes_fwd"] - 2 * per_seq_states == 2054 * th  # q k v o 1024, g 4, beta 2, h 1024
    assert m["bytes_bwd"] - 2 * per_seq_states == (7 * 256 + 4 + 4 + 2 + 2 + 1024) * th


def test_partial_chunks_count_their_own_length():
    # a 65-token sequence is one full chunk and one chunk of 1 token: the flops are the sum of
    # the two chunk terms, not two full chunks
    import bench
    from chunked_gated_delta_04_gb300.inputs import Workload
    import torch

    w = Workload("x", torch.bfloat16, 1, 65, 1, 1, 128, 128)
    inp = {"seqlens": [65], "num_seqs": 1, "S0": None, "dS_T": None}
    m = bench.work_model(inp, w)
    full, one = bench.work_model({**inp, "seqlens": [64]}, w), bench.work_model({**inp, "seqlens": [1]}, w)
    assert m["flops_fwd"] == pytest.approx(full["flops_fwd"] + one["flops_fwd"])
    assert m["flops_bwd"] == pytest.approx(full["flops_bwd"] + one["flops_bwd"])
    assert m["tensor_bytes"]["h_saved"] == 2 * 128 * 128 * 4


def test_ncu_traffic_is_reported_only_for_unchanged_sources():
    import bench

    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    lines = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    assert lines, "no traffic entries"
    for stage, nbytes, digest, src in lines:
        with open(os.path.join(ROOT, "chunked_gated_delta_04_gb300", "csrc", src), "rb") as f:
            current = hashlib.sha256(f.read()).hexdigest()[:16]
        got = bench.ncu_traffic(stage)
        if current == digest:
            assert got == float(nbytes)
        else:
            assert got is None


def test_saved_factors_leave_the_recompute_out_of_the_backward_flops():
    # with the forward's chunk factors saved the backward does not form W = T' K (2 c^2 DK),
    # U = T'' V (2 c^2 DV) or the inverse (c^3 / 3): at c = 64, D = 128 that is 2.18 MFLOP less
    # per chunk-head, 34.1 kFLOP less per token-head (476.5 -> 442.4 kFLOP)
    import bench

    m, w = _model("b2_t4096")
    inp = {"seqlens": [w.T] * w.B, "num_seqs": w.B, "S0": object(), "dS_T": object()}
    ms = bench.work_model(inp, w, save_wy=True)
    th = w.B * w.T * w.Hv
    per_chunk = 2 * 64 * 64 * 128 * 2 + 64 ** 3 / 3
    assert (m["flops_bwd"] - ms["flops_bwd"]) / th == pytest.approx(per_chunk / 64, rel=1e-12)
    assert ms["flops_bwd"] / th == pytest.approx(442.4e3, rel=2e-4)
    assert ms["flops_fwd"] == m["flops_fwd"] and ms["bytes_bwd"] == m["bytes_bwd"]
