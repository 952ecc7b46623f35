"""Host-side tests of the C ABI (no GPU needed): the library loads, exports every
function declared in include/gdr.h, sizes its buffers correctly and rejects bad
arguments with a status code before launching anything."""
import ctypes
import os
import re

import pytest
import torch

import chunked_gated_delta_04_gb300 as gdr
from chunked_gated_delta_04_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gdr.load()


def declared_functions():
    hdr = open(os.path.join(ROOT, "include", "gdr.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return sorted(set(re.findall(r"\b(gdr_[a-z0-9_]+)\s*\(", hdr)))


def test_library_exports_every_declared_function(lib):
    names = declared_functions()
    assert "gdr_fwd" in names and "gdr_bwd" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(gdr.EXPORTS)


def prob(**kw):
    args = dict(B=2, T=130, Hk=2, Hv=4, DK=64, DV=32, dtype=torch.bfloat16, layout="KV")
    args.update(kw)
    return gdr.make_problem(**args)


def test_size_queries(lib):
    p = prob()
    assert gdr.gdr_max_chunks(p) == 2 * 3
    assert gdr.gdr_saved_states_bytes(p) == 6 * 4 * 64 * 32 * 4
    assert gdr.gdr_fwd_workspace_bytes(p) > 0
    assert gdr.gdr_bwd_workspace_bytes(p) > gdr.gdr_fwd_workspace_bytes(p)
    # varlen bound: floor(T/64) + num_seqs
    cu = torch.tensor([0, 1, 65, 300], dtype=torch.int32)
    pv = gdr.make_problem(1, 300, 1, 1, 32, 32, torch.float32, "VK", cu_seqlens=cu)
    assert gdr.gdr_max_chunks(pv) == 300 // 64 + 3
    assert gdr.gdr_path(prob(DK=128, DV=128)) in (0, 1)
    assert gdr.gdr_path(prob(dtype=torch.float32)) == 0
    # bf16 saved states: half the bytes, same workspaces
    assert gdr.gdr_saved_states_bytes(prob(h_dtype=torch.bfloat16)) == 6 * 4 * 64 * 32 * 2
    assert gdr.gdr_fwd_workspace_bytes(prob(h_dtype=torch.bfloat16)) == gdr.gdr_fwd_workspace_bytes(p)
    # the fused prologue keeps its mapped inputs in the workspace
    assert gdr.gdr_fwd_workspace_bytes(prob(prologue=7)) > gdr.gdr_fwd_workspace_bytes(p)
    assert gdr.gdr_bwd_workspace_bytes(prob(prologue=1)) > gdr.gdr_bwd_workspace_bytes(p)
    # saved factors: on the tensor-core path 49408 bytes per (chunk, v-head) move from the
    # workspaces into the saved buffer; on the SIMT path with DK, DV <= 64 fp32 gamma, W^T, T,
    # K K^T * Gam, P^T and Vn (each region 256-byte aligned); larger SIMT heads save nothing
    def a256(x):
        return (x + 255) // 256 * 256
    chH = 6 * 4
    factors = (a256(chH * 64 * 4) + a256(chH * 64 * 64 * 4) + 3 * a256(chH * 64 * 64 * 4) +
               a256(chH * 64 * 32 * 4))
    assert gdr.gdr_saved_states_bytes(prob(save_wy=True)) == a256(gdr.gdr_saved_states_bytes(p)) + factors
    assert gdr.gdr_saved_states_bytes(prob(DK=96, DV=96, save_wy=True)) == gdr.gdr_saved_states_bytes(prob(DK=96, DV=96))
    pt, pts = prob(DK=128, DV=128), prob(DK=128, DV=128, save_wy=True)
    chH = 6 * 4
    if gdr.gdr_path(pt) == 1:
        assert gdr.gdr_saved_states_bytes(pts) == gdr.gdr_saved_states_bytes(pt) + chH * 49408
        assert gdr.gdr_fwd_workspace_bytes(pts) < gdr.gdr_fwd_workspace_bytes(pt)
        assert gdr.gdr_bwd_workspace_bytes(pts) < gdr.gdr_bwd_workspace_bytes(pt)
    else:
        assert gdr.gdr_saved_states_bytes(pts) == gdr.gdr_saved_states_bytes(pt)
        assert gdr.gdr_fwd_workspace_bytes(pts) == gdr.gdr_fwd_workspace_bytes(pt)


@pytest.mark.parametrize("kw,code", [
    (dict(Hv=3), gdr.GDR_ERR_INVALID_ARG),          # Hv % Hk != 0
    (dict(DK=72), gdr.GDR_ERR_UNSUPPORTED),         # not a multiple of 16
    (dict(DV=256), gdr.GDR_ERR_UNSUPPORTED),        # wider than 128
    (dict(layout=7), gdr.GDR_ERR_INVALID_ARG),
    (dict(dtype=torch.float16), gdr.GDR_ERR_INVALID_ARG),
    (dict(T=-1), gdr.GDR_ERR_INVALID_ARG),
    (dict(h_dtype=torch.float16), gdr.GDR_ERR_INVALID_ARG),  # h_saved is fp32 or bf16
    (dict(prologue=8), gdr.GDR_ERR_INVALID_ARG),              # unknown prologue bit
    (dict(save_wy=2), gdr.GDR_ERR_INVALID_ARG),               # save_wy is 0 or 1
    (dict(cp_fwd=-2), gdr.GDR_ERR_INVALID_ARG),               # context-parallel segments: -1 (auto), 0 .. 64
    (dict(cp_bwd=65), gdr.GDR_ERR_INVALID_ARG),
    # 2^30 token-heads but 2^24 chunk-heads: the saved states' 128-row blocks would pass 2^31
    (dict(T=1 << 27), gdr.GDR_ERR_UNSUPPORTED),
])
def test_bad_problems_are_rejected(lib, kw, code):
    p = prob(**kw)
    fake = 1 << 20  # never dereferenced: validation fails first
    st = gdr.gdr_fwd(p, fake, fake, fake, fake, fake, None, fake, None, fake, fake, workspace_bytes=1 << 30,
                     stream=0)
    assert st == code
    assert gdr.gdr_max_chunks(p) == 0


def test_context_parallel_workspace(lib):
    # off (0 or 1) costs nothing; P segments add three [num_seqs][Hv][P][128][128] fp32 matrices
    # per direction on the tensor-core path (the SIMT path ignores the setting)
    p = prob(DK=128, DV=128)
    for cp in (0, 1):
        assert gdr.gdr_fwd_workspace_bytes(prob(DK=128, DV=128, cp_fwd=cp)) == gdr.gdr_fwd_workspace_bytes(p)
    pf, pb = prob(DK=128, DV=128, cp_fwd=4), prob(DK=128, DV=128, cp_bwd=3)
    mats = 2 * 4 * 128 * 128 * 4
    if gdr.gdr_path(p) == 1:
        assert gdr.gdr_fwd_workspace_bytes(pf) == gdr.gdr_fwd_workspace_bytes(p) + 3 * 4 * mats
        assert gdr.gdr_bwd_workspace_bytes(pf) == gdr.gdr_bwd_workspace_bytes(p)
        assert gdr.gdr_bwd_workspace_bytes(pb) == gdr.gdr_bwd_workspace_bytes(p) + 3 * 3 * mats
    else:
        assert gdr.gdr_fwd_workspace_bytes(pf) == gdr.gdr_fwd_workspace_bytes(p)
        assert gdr.gdr_bwd_workspace_bytes(pb) == gdr.gdr_bwd_workspace_bytes(p)
    assert gdr.gdr_fwd_workspace_bytes(prob(cp_fwd=8)) == gdr.gdr_fwd_workspace_bytes(prob())  # SIMT shape
    # the resolved counts: explicit values pass through on the tensor-core path, the SIMT path has none
    if gdr.gdr_path(p) == 1:
        assert gdr.gdr_debug_cp_segments(prob(DK=128, DV=128, cp_fwd=4, cp_bwd=0)) == (4, 1)
    assert gdr.gdr_debug_cp_segments(prob(cp_fwd=4, cp_bwd=4)) == (1, 1)
    assert gdr.gdr_debug_cp_segments(prob(DK=128, DV=128, cp_fwd=gdr.GDR_CP_AUTO, cp_bwd=1))[1] == 1


def test_context_parallel_split_matches_the_oracle(lib):
    """The library's segment split is the oracle's (sizes within one, the longer ones first,
    clamped to the chunk count, one empty segment for an empty sequence)."""
    from oracle.context_parallel import split_chunks
    for nc in [0, 1, 2, 7, 14, 64, 1024, 1031]:
        for P in [1, 2, 3, 4, 5, 8, 14, 16, 64]:
            want = split_chunks(nc, P)
            c0 = 5  # a sequence whose first chunk is global chunk 5
            got = []
            nseg = gdr.gdr_debug_cp_segment(c0, c0 + nc, P, 0)[2]
            assert nseg == max(1, min(P, nc))
            for s in range(nseg):
                lo, hi, n2 = gdr.gdr_debug_cp_segment(c0, c0 + nc, P, s)
                assert n2 == nseg
                if hi > lo:
                    got.append((lo - c0, hi - c0))
            assert got == want, (nc, P, got, want)
            assert gdr.gdr_debug_cp_segment(c0, c0 + nc, P, nseg) == (c0 + nc, c0 + nc, nseg)
    with pytest.raises(ValueError):
        gdr.gdr_debug_cp_segment(0, 10, 0, 0)


def test_largest_accepted_chunk_count(lib):
    # one chunk fewer per sequence than the rejected case above: 2^24 - 8 chunk-heads
    p = prob(T=(1 << 27) - 64)
    assert gdr.gdr_max_chunks(p) == 2 * ((1 << 21) - 1)


def test_pointer_and_workspace_checks(lib):
    p = prob()
    a = 1 << 20
    ws_bytes = gdr.gdr_fwd_workspace_bytes(p)
    # null required pointer
    assert gdr.gdr_fwd(p, None, a, a, a, a, None, a, None, a, a, ws_bytes, 0) == gdr.GDR_ERR_INVALID_ARG
    # misaligned pointer
    assert gdr.gdr_fwd(p, a + 4, a, a, a, a, None, a, None, a, a, ws_bytes, 0) == gdr.GDR_ERR_ALIGNMENT
    # workspace too small / missing / misaligned
    assert gdr.gdr_fwd(p, a, a, a, a, a, None, a, None, a, a, ws_bytes - 1, 0) == gdr.GDR_ERR_WORKSPACE
    assert gdr.gdr_fwd(p, a, a, a, a, a, None, a, None, a, None, ws_bytes, 0) == gdr.GDR_ERR_WORKSPACE
    assert gdr.gdr_fwd(p, a, a, a, a, a, None, a, None, a, a + 128, ws_bytes, 0) == gdr.GDR_ERR_ALIGNMENT
    wb = gdr.gdr_bwd_workspace_bytes(p)
    args = [a] * 6 + [a, None] + [a] * 5 + [None]
    assert gdr.gdr_bwd(p, *args, a, wb - 1, 0) == gdr.GDR_ERR_WORKSPACE
    args[6] = None  # dO
    assert gdr.gdr_bwd(p, *args, a, wb, 0) == gdr.GDR_ERR_INVALID_ARG
    # varlen needs B == 1
    cu = torch.tensor([0, 5, 10], dtype=torch.int32)
    pv = gdr.make_problem(2, 10, 1, 1, 32, 32, torch.float32, "KV", cu_seqlens=cu)
    assert gdr.gdr_fwd(pv, a, a, a, a, a, None, a, None, a, a, 1 << 30, 0) == gdr.GDR_ERR_INVALID_ARG


def test_status_strings(lib):
    for s in range(7):
        assert gdr.gdr_status_string(s).startswith("GDR_")


def test_saved_buffer_helpers(lib):
    # the binding's saved buffer: a states view whose storage also holds the saved factors;
    # a buffer too small for the problem is refused on the host before any call
    for save_wy in (False, True):
        p = prob(DK=128, DV=128, save_wy=save_wy)
        h = gdr.alloc_saved(p, torch.float32, "cpu")
        assert tuple(h.shape) == (gdr.gdr_max_chunks(p), p.Hv, 128, 128) and h.dtype == torch.float32
        assert h.untyped_storage().nbytes() >= gdr.gdr_saved_states_bytes(p)
        gdr._check_saved(p, h)
    p = prob(DK=128, DV=128, save_wy=True)
    small = torch.empty((gdr.gdr_max_chunks(p), p.Hv, 128, 128), dtype=torch.float32)
    if gdr.gdr_saved_states_bytes(p) > small.untyped_storage().nbytes():  # tensor-core path
        with pytest.raises(ValueError):
            gdr._check_saved(p, small)
    hb = gdr.alloc_saved(prob(h_dtype=torch.bfloat16), torch.bfloat16, "cpu")
    assert hb.dtype == torch.bfloat16
