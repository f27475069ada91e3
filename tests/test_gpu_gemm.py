"""The tcgen05 GEMM core against a CPU fp32 matmul, all four operand layouts."""
import pytest
import torch

from gpu_util import need_gpu, rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("a_layout,b_layout", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 256, 512), (200, 128, 192), (384, 64, 128),
                                   (1000, 512, 1024)])
def test_dense_gemm_matches_fp32_matmul(a_layout, b_layout, M, N, K):
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import binding as B
    g = torch.Generator().manual_seed(M * 7 + N * 3 + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    Bm = torch.randn(N, K, generator=g).to(torch.bfloat16)
    a_store = (A if a_layout == 0 else A.t().contiguous()).cuda()
    b_store = (Bm if b_layout == 0 else Bm.t().contiguous()).cuda()
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_gemm_bf16(a_store, b_store, C, M, N, K, a_layout, b_layout, status)
    assert B.moe_check_status(status) == 0
    ref = A.float() @ Bm.float().T
    assert rel_err(C.float().cpu().numpy(), ref.double().numpy()) < 1e-2


@pytest.mark.parametrize("a_layout,b_layout", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (256, 128, 512), (200, 256, 192), (384, 128, 128),
                                   (1000, 512, 1024), (128, 256, 256)])
def test_pair_gemm_matches_fp32_matmul(a_layout, b_layout, M, N, K):
    """The CTA-pair kernel (M = 256 per MMA), including a lone 128-row tile and ragged M."""
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import binding as B
    g = torch.Generator().manual_seed(M * 5 + N * 3 + K + 17)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    Bm = torch.randn(N, K, generator=g).to(torch.bfloat16)
    a_store = (A if a_layout == 0 else A.t().contiguous()).cuda()
    b_store = (Bm if b_layout == 0 else Bm.t().contiguous()).cuda()
    C = torch.full((M + 64, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_gemm_bf16_pair(a_store, b_store, C, M, N, K, a_layout, b_layout, status)
    assert B.moe_check_status(status) == 0
    ref = A.float() @ Bm.float().T
    assert rel_err(C[:M].float().cpu().numpy(), ref.double().numpy()) < 1e-2
    assert torch.isnan(C[M:].float()).all()          # nothing written past row M
