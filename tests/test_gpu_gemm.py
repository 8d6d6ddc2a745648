"""The tcgen05 GEMM core in isolation (test-only entry flce_debug_gemm).

D = A B^T for every operand layout the loss path uses: K-major A and B (the
logit GEMM), MN-major A and B (the dW GEMM), K-major A with MN-major B (the dX
GEMM), plus MN-major A with K-major B, for both tile shapes (CTA-pair 256 x 256 and
single-CTA 128 x 256).  Checked against a float64 product of the same bf16
values.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

SHAPES = [
    (128, 256, 64),     # one tile, one k-block
    (304, 520, 200),    # ragged M, N and K tails
    (1024, 768, 1024),  # several tiles per CTA, long K
]


@pytest.fixture(params=[1, 0], ids=["cta_pair", "single_cta"], autouse=True)
def tile_shape(request):
    from linear_cross_entropy_logit_gb300 import binding as B
    B.flce_set_cta_pair(request.param)
    yield request.param
    B.flce_set_cta_pair(1)


def _bf16(rng, shape):
    import torch
    return torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (1, 1), (0, 1), (1, 0)])
@pytest.mark.parametrize("M,Nn,K", SHAPES)
def test_debug_gemm(a_mn, b_mn, M, Nn, K):
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    rng = np.random.default_rng(M * 7 + Nn * 3 + K + 11 * a_mn + 13 * b_mn)
    A = _bf16(rng, (M, K))   # logical A: M x K
    Bm = _bf16(rng, (Nn, K))  # logical B: Nn x K
    want = A.double() @ Bm.double().T
    A_st = A.T.contiguous() if a_mn else A.contiguous()
    B_st = Bm.T.contiguous() if b_mn else Bm.contiguous()
    D, err = B.flce_debug_gemm(A_st.cuda(), B_st.cuda(), M, Nn, K, bool(a_mn), bool(b_mn))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = D.cpu().double()
    rel = (got - want).norm() / want.norm()
    assert rel < 1e-5, f"rel Frobenius error {rel:.3e}"
    assert torch.isfinite(got).all()


def test_debug_gemm_accumulate():
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    rng = np.random.default_rng(5)
    M, Nn, K = 256, 512, 192
    A, Bm = _bf16(rng, (M, K)), _bf16(rng, (Nn, K))
    D0 = torch.from_numpy(rng.standard_normal((M, Nn)).astype(np.float32))
    D = D0.clone().cuda()
    B.flce_debug_gemm(A.cuda(), Bm.T.contiguous().cuda(), M, Nn, K, False, True, D=D,
                      accumulate=True)
    torch.cuda.synchronize()
    want = D0.double() + A.double() @ Bm.double().T
    rel = (D.cpu().double() - want).norm() / want.norm()
    assert rel < 1e-5
