"""The tcgen05 GEMM engine (TMA-fed, TMEM accumulators) through its C-ABI test
hook, against a float64 product of the same bf16 inputs.  Covers K-major and
MN-major operands, ragged M/N/K, bias and accumulate."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _ref(A, B, M, N, K, a_mn, b_mn, bias, D0):
    a = (A[:K, :M].t() if a_mn else A[:M, :K]).double().cpu()
    b = (B[:K, :N].t() if b_mn else B[:N, :K]).double().cpu()
    r = a @ b.t()
    if bias is not None:
        r = r + bias.double().cpu()
    if D0 is not None:
        r = r + D0.double().cpu()
    return r


def _pad8(n):
    return (n + 7) // 8 * 8


@pytest.mark.parametrize("a_mn", [0, 1])
@pytest.mark.parametrize("b_mn", [0, 1])
@pytest.mark.parametrize("MNK", [(128, 256, 64), (300, 520, 200), (77, 96, 136), (1, 64, 8), (640, 128, 1000)])
def test_gemm_matches_float64(a_mn, b_mn, MNK):
    from recurrent_neural_network_gb300 import rnn
    M, N, K = MNK
    g = torch.Generator().manual_seed(M * 7 + N * 3 + K + a_mn + 2 * b_mn)
    dev = "cuda"
    A = (torch.randn(K, _pad8(M), generator=g) if a_mn else torch.randn(M, _pad8(K), generator=g)).to(torch.bfloat16)
    B = (torch.randn(K, _pad8(N), generator=g) if b_mn else torch.randn(N, _pad8(K), generator=g)).to(torch.bfloat16)
    bias = torch.randn(N, generator=g)
    Ad, Bd, biasd = A.to(dev), B.to(dev), bias.to(dev)
    D = torch.full((M, N), float("nan"), device=dev)
    rnn.gemm_bf16(Ad, Bd, D, M, N, K, A.shape[1], B.shape[1], N, a_mn=a_mn, b_mn=b_mn, bias=biasd)
    torch.cuda.synchronize()
    ref = _ref(A, B, M, N, K, a_mn, b_mn, bias, None)
    err = (D.double().cpu() - ref).abs().max().item()
    assert err <= 1e-5 * K ** 0.5 * 4 + 1e-5, err
    # accumulate into the result
    D0 = D.clone()
    rnn.gemm_bf16(Ad, Bd, D, M, N, K, A.shape[1], B.shape[1], N, a_mn=a_mn, b_mn=b_mn, accumulate=True)
    torch.cuda.synchronize()
    ref2 = _ref(A, B, M, N, K, a_mn, b_mn, None, D0)
    err2 = (D.double().cpu() - ref2).abs().max().item()
    assert err2 <= 2e-5 * K ** 0.5 * 4 + 1e-5, err2


def test_gemm_large_persistent_grid():
    """More tiles than SMs: the persistent tile loop and the TMEM double buffer."""
    from recurrent_neural_network_gb300 import rnn
    M, N, K = 2048, 4096, 512
    g = torch.Generator().manual_seed(5)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    D = torch.empty(M, N, device="cuda")
    rnn.gemm_bf16(A.cuda(), B.cuda(), D, M, N, K, K, K, N)
    torch.cuda.synchronize()
    ref = A.double() @ B.double().t()
    assert (D.double().cpu() - ref).abs().max().item() < 2e-3
