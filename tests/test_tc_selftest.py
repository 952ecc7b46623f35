"""Device check of the tcgen05 operand layouts (K-major / MN-major, 128-byte swizzle,
TMEM read-back) against a torch matmul, before the tensor-core kernels rely on them."""
import pytest
import torch

import chunked_gated_delta_04_gb300 as gdr

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N", [64, 128])
@pytest.mark.parametrize("K", [64, 128])
@pytest.mark.parametrize("a_mn", [0, 1])
@pytest.mark.parametrize("b_mn", [0, 1])
def test_tc_gemm_layouts(N, K, a_mn, b_mn):
    g = torch.Generator(device="cpu").manual_seed(N * 7 + K * 3 + a_mn * 2 + b_mn)
    Am = torch.randn(128, K, generator=g).bfloat16()
    Bm = torch.randn(K, N, generator=g).bfloat16()
    A = (Am.t() if a_mn else Am).contiguous().cuda()
    B = (Bm if b_mn else Bm.t()).contiguous().cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert gdr.gdr_debug_tc_gemm(A, B, D, N, K, a_mn, b_mn, status) == 0
    torch.cuda.synchronize()
    assert status.item() == 0
    ref = Am.float() @ Bm.float()
    err = (D.cpu() - ref).abs().max().item()
    assert err < 1e-3 * ref.abs().max().item(), err
