"""The GEMM building block of the projection (key design 3 of
"Communication-Efficient LLM Adaptation over Decentralized GPU Meshes"):
C = A B^T on the tcgen05 TF32 path and on the fp32 SIMT path.

Small integers are exact in TF32 and their products and sums are exact in
fp32, so on such inputs both paths must match the float64 product exactly: any
layout, swizzle or descriptor mistake shows up as a wrong value.  Random
normal inputs check the TF32 rounding error bound."""
import numpy as np
import pytest
import torch

import spectral_corrected_optimizer_gb300 as so
from gpu_util import ensure_lib

pytestmark = pytest.mark.gpu

SHAPES = [(128, 256, 32), (256, 512, 64), (300, 520, 200), (1, 8, 4), (129, 257, 36), (100, 300, 20),
          (2048, 2048, 2048), (8192, 2048, 512), (512, 4096, 100)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


@pytest.mark.parametrize("prec", [so.PREC_TF32, so.PREC_FP32])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_exact_on_small_integers(prec, M, N, K):
    g = torch.Generator().manual_seed(M * 7 + N * 3 + K)
    A = torch.randint(-4, 5, (M, K), generator=g).float()
    B = torch.randint(-4, 5, (N, K), generator=g).float()
    C = so.gemm_nt(A.cuda(), B.cuda(), prec)
    want = (A.double() @ B.double().T).float()
    assert torch.equal(C.cpu(), want)


@pytest.mark.parametrize("M,N,K", SHAPES[:6])
def test_tf32_error_bound(M, N, K):
    g = torch.Generator().manual_seed(1)
    A = torch.randn(M, K, generator=g)
    B = torch.randn(N, K, generator=g)
    C = so.gemm_nt(A.cuda(), B.cuda(), so.PREC_TF32).cpu().double()
    ref = A.double() @ B.double().T
    bound = (A.double().abs() @ B.double().abs().T) * 2.0 ** -9 + 1e-6
    assert ((C - ref).abs() <= bound).all()
    assert (C - ref).norm() / ref.norm() <= 2e-3


def test_tf32_rejects_unsupported_layout():
    A = torch.zeros(16, 6, device="cuda")
    B = torch.zeros(8, 6, device="cuda")
    with pytest.raises(so.SpecOptimError) as e:
        so.gemm_nt(A, B, so.PREC_TF32)
    assert e.value.code == so.ERR_NOT_IMPLEMENTED
    # the SIMT path takes any layout
    assert so.gemm_nt(A, B, so.PREC_FP32).abs().sum().item() == 0
