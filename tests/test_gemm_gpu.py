"""GPU checks of the tcgen05 bf16 GEMM against a plain PyTorch fp64 CPU matmul of the same bf16
operands, for all four operand layouts, tile multiples and ragged edges."""
import pytest
import torch

from shared_prefix_grouped_gb300 import api
from shared_prefix_grouped_gb300.build import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()


@pytest.mark.parametrize("a_mn", [False, True])
@pytest.mark.parametrize("b_mn", [False, True])
@pytest.mark.parametrize("mnk", [(128, 128, 64), (256, 384, 512), (200, 136, 72), (8, 1000, 1032)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gemm_matches_fp64(a_mn, b_mn, mnk, out_dtype):
    M, N, K = mnk
    g = torch.Generator().manual_seed(M * 7 + N * 3 + K)
    A = torch.randn((M, K), generator=g).to(torch.bfloat16)
    B = torch.randn((N, K), generator=g).to(torch.bfloat16)
    ref = A.double() @ B.double().T
    a_st = A.T.contiguous() if a_mn else A
    b_st = B.T.contiguous() if b_mn else B
    # MN-major operands need their contiguous dimension to be a multiple of 8 (16-byte rows)
    if (a_mn and M % 8) or (b_mn and N % 8):
        pytest.skip("leading dimension not a multiple of 8")
    C = api.gemm_bf16(a_st.cuda(), b_st.cuda(), a_mn=a_mn, b_mn=b_mn, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert api.device_status() == 0
    err = (C.double().cpu() - ref).abs().max().item() / ref.abs().max().item()
    tol = 1e-5 if out_dtype == torch.float32 else 1e-2
    assert err < tol, err
