"""The tcgen05 head contraction alone (rl_gemm_bf16_tn) against a plain PyTorch fp32
matmul of the same bf16 values: tiles, K blocks, ragged M/N tails."""
import pytest
import torch

import lm_head_gb300 as rh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_gb300 import build
    build.build()
    rh.load()


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 128), (300, 1000, 192), (129, 260, 2048),
                                   (1024, 4096, 2048), (77, 24, 8)])
def test_gemm_matches_fp32_reference(M, N, K):
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N * 3 + K)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, device="cuda", generator=g).to(torch.bfloat16)
    D, st = rh.rl_gemm_bf16_tn(A, B)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = A.double() @ B.double().T
    err = (D.double() - ref).abs().max().item()
    assert err <= 1e-5 * (K ** 0.5) * max(1.0, ref.abs().max().item()), err


@pytest.mark.parametrize("a_mn,b_mn", [(0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (296, 1000, 192), (1024, 2048, 2048), (136, 24, 40)])
def test_gemm_mn_major_operands(M, N, K, a_mn, b_mn):
    """Operands stored M/N-contiguous ([K, M], [K, N]) read without a transpose."""
    g = torch.Generator(device="cuda").manual_seed(M + 11 * N + 7 * K + a_mn + 2 * b_mn)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, device="cuda", generator=g).to(torch.bfloat16)
    Aop = A.T.contiguous() if a_mn else A
    Bop = B.T.contiguous() if b_mn else B
    D, st = rh.rl_gemm_bf16(Aop, bool(a_mn), Bop, bool(b_mn))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = A.double() @ B.double().T
    err = (D.double() - ref).abs().max().item()
    assert err <= 1e-5 * (K ** 0.5) * max(1.0, ref.abs().max().item()), err


def test_gemm_rejects_unaligned_contiguous_extent():
    A = torch.zeros(192, 300, device="cuda", dtype=torch.bfloat16)   # [K, M] with M % 8 != 0
    B = torch.zeros(1000, 192, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(rh.RLHeadError):
        rh.rl_gemm_bf16(A, True, B, False)
