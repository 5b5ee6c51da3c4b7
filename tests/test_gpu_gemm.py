"""The tcgen05 GEMM core alone, for each operand majorness and each tile
shape (one CTA per 128 x 256 tile, a CTA pair per 256 x 256 tile, two pairs
per 512 x 256 tile, a pair per 256 x 512 tile), against the float64 product
of the same bf16 operands; and the bounded device wait."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=["single", "pair", "wide"])
def handle(request):
    from linear_cross_entropy_token_gb300 import FLCE
    h = FLCE("bf16", 0, cta=request.param)
    yield h
    h.close()


SHAPES = [(128, 256, 64), (256, 512, 192), (200, 296, 136), (384, 768, 1024), (64, 40, 8),
          (520, 264, 320)]


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)],
                         ids=["A_K-B_K", "A_K-B_MN", "A_MN-B_MN", "A_MN-B_K"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_core(handle, a_mn, b_mn, M, N, K):
    g = torch.Generator().manual_seed(M * 7 + N * 3 + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)   # logical A (M x K)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)   # logical B (N x K)
    ref = (A.double() @ B.double().T).numpy()
    Ad = (A.T.contiguous() if a_mn else A).cuda()
    Bd = (B.T.contiguous() if b_mn else B).cuda()
    C = handle.check_gemm(Ad, Bd, bool(a_mn), bool(b_mn), M, N, K).double().cpu().numpy()
    err = np.linalg.norm(C - ref) / np.linalg.norm(ref)
    if err > 1e-5:
        # where the product is wrong tells a layout mistake apart
        bad = ~np.isclose(C, ref, rtol=1e-3, atol=1e-2)
        rows = np.flatnonzero(bad.any(axis=1))
        cols = np.flatnonzero(bad.any(axis=0))
        pytest.fail(f"relative error {err:.3e}; wrong rows {rows[:8]}..{rows[-4:]} "
                    f"({len(rows)}), wrong cols {cols[:8]}..{cols[-4:]} ({len(cols)}); "
                    f"C[0,:4]={C[0, :4]}, ref[0,:4]={ref[0, :4]}")


def test_bounded_wait_reports_timeout(handle):
    """A device-side wait on a barrier nothing completes gives up after its
    limit, reports FLCE_ERR_TIMEOUT, and leaves the context usable."""
    st = handle.check_wait_timeout(2000)   # 2 ms
    assert st == 5
    # the context still works afterwards
    A = torch.ones(128, 64, dtype=torch.bfloat16, device="cuda")
    B = torch.ones(256, 64, dtype=torch.bfloat16, device="cuda")
    C = handle.check_gemm(A, B, False, False, 128, 256, 64)
    assert torch.all(C == 64.0)
