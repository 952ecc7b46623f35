"""Delay injection: the kernels' hand-offs between roles hold when one role runs late.

libgdr_delay.so is the same source built with -DGDR_DEBUG_DELAY: at each hand-off point one
role sleeps a short, bounded, pseudo-random time (the copy threads before their TMA loads, one
warp of an epilogue before its shared-memory writes, the MMA-issuing thread before a product,
the reverse walk and the fused forward's prep role before publishing a chunk's flag, one CTA of
each cluster pair before sending its half of dq/dk).  Only the timing changes, and the results
do not depend on it (no floating-point atomics, fixed reduction orders), so every output must
equal the normal build's bit for bit.  A missing wait or barrier that the normal timing happens
to cover shows up here as a difference.  Every wait in the kernels stays bounded, and the
sleeps are microseconds against limits of seconds: nothing here can hang or fault the GPU.

The cases cover each kernel family: the fused backward (walk + gradients in one cooperative
launch) at the benchmark's B=2, T=4096, H=16 shape; the fused forward (few long chains);
variable length; Hv = 2 Hk (cluster-pair gradients); Hv = 4 Hk (partials + reduce); more state
CTAs than SMs (single-buffered forward state); context-parallel segments (first-pass maps, the
boundary scan with its bulk copies, the fused kernel's second pass; fixed and variable length).
"""
import pytest
import torch

import chunked_gated_delta_04_gb300 as gdr
from chunked_gated_delta_04_gb300 import build as gbuild
from chunked_gated_delta_04_gb300.inputs import make_inputs, small_workload
from gdr_testlib import run_gpu

pytestmark = pytest.mark.gpu

CASES = [
    # name, B, T, Hk, Hv, seqlens, layout, save_wy, context-parallel segments (fwd, bwd)
    ("fused_bwd_b2_t4096", 2, 4096, 16, 16, None, "KV", True, (1, 1)),
    ("fused_fwd_few_chains", 1, 2048, 2, 2, None, "VK", True, (1, 1)),
    ("varlen", 1, None, 4, 4, [0, 70, 130, 1, 200, 64, 1500], "KV", False, (1, 1)),
    ("pair_gva", 2, 512, 2, 4, None, "KV", True, (1, 1)),
    ("group_gva4", 1, 300, 1, 4, None, "VK", False, (1, 1)),
    ("single_buffered_state", 3, 200, 13, 13, None, "KV", True, (1, 1)),
    ("cp_fixed", 1, 3000, 2, 2, None, "KV", True, (5, 7)),
    ("cp_varlen", 1, None, 1, 2, [900, 64, 1300], "VK", False, (3, 4)),
]


@pytest.fixture(scope="module")
def delay_lib():
    return gbuild.build(delay=True)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_delayed_roles_give_bitwise_identical_results(delay_lib, case):
    name, B, T, Hk, Hv, lens, layout, save_wy, (cp_f, cp_b) = case
    if lens is None:
        w = small_workload(name, torch.bfloat16, B=B, T=T, Hk=Hk, Hv=Hv, DK=128, DV=128, layout=layout)
    else:
        w = small_workload(name, torch.bfloat16, Hk=Hk, Hv=Hv, DK=128, DV=128, seqlens=lens, layout=layout)
    inp = make_inputs(w)
    ref = run_gpu(inp, save_wy=save_wy, cp_fwd=cp_f, cp_bwd=cp_b)
    torch.cuda.synchronize()
    with gdr.library(delay_lib):
        for _ in range(2):  # two runs: the sleeps differ between them
            got = run_gpu(inp, save_wy=save_wy, cp_fwd=cp_f, cp_bwd=cp_b)
            torch.cuda.synchronize()
            for key, t in ref.items():
                if t is None:
                    continue
                if key == "h_saved" and lens is not None:  # slots past the last real chunk: unwritten
                    n = sum((L + 63) // 64 for L in lens)
                    assert torch.equal(got[key][:n], t[:n]), f"{name}: {key}"
                else:
                    assert torch.equal(got[key], t), f"{name}: {key}"
