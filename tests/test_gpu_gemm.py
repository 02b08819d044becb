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
