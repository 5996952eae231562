"""The tcgen05 GEMM core (C ABI diagnostic mtp_gemm_bf16) against a plain
PyTorch fp32 reference of the same product, shapes spanning several tiles
with ragged M, N and K tails."""
import pytest
import torch

from deepseek_sequential_mtp_gb300 import lib

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 256), (300, 1000, 200),
                                   (1024, 3072, 1024), (777, 1536, 2816), (8192, 1024, 2048)])
def test_gemm_matches_fp32_reference(M, N, K):
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, device="cuda", generator=g).to(torch.bfloat16)
    C = lib.gemm_bf16(A, B)
    lib.check_errors()
    ref = A.float() @ B.float().T
    err = (C.float() - ref).abs()
    # one bf16 rounding of the fp32 result (2^-8 relative) plus accumulation order
    tol = ref.abs() * 2 ** -8 + 1e-3 * K ** 0.5
    assert bool((err <= tol).all()), f"max err {err.max().item()}"


def test_gemm_repeated_calls_stable():
    A = torch.randn(512, 512, device="cuda").to(torch.bfloat16)
    B = torch.randn(768, 512, device="cuda").to(torch.bfloat16)
    C0 = lib.gemm_bf16(A, B)
    for _ in range(20):
        C1 = lib.gemm_bf16(A, B)
    torch.cuda.synchronize()
    assert torch.equal(C0, C1)
    assert lib.check_errors() == 0


@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (True, False), (False, True), (True, True)])
@pytest.mark.parametrize("M,N,K,splits", [(128, 256, 64, 1), (296, 1000, 200, 1), (1024, 512, 8192, 4),
                                          (200, 776, 1000, 2)])
def test_f32acc_operand_layouts(a_mn, b_mn, M, N, K, splits):
    """out += A B^T into fp32 with either operand read K-major or MN-major
    (the transpose of a row-major matrix, as the training step's weight and
    input gradients use): against the fp32 product of the same bf16 values."""
    g = torch.Generator(device="cuda").manual_seed(M + 3 * N + K)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, device="cuda", generator=g).to(torch.bfloat16)
    out0 = torch.randn(M, N, device="cuda", generator=g)
    out = out0.clone()
    lib.gemm_f32acc(A.t().contiguous() if a_mn else A, B.t().contiguous() if b_mn else B, out, a_mn=a_mn, b_mn=b_mn,
                    splits=splits)
    lib.check_errors()
    ref = out0.double() + A.double() @ B.double().T
    err = (out.double() - ref).abs()
    tol = 1e-5 * (A.double().abs() @ B.double().abs().T) + 1e-5 * out0.double().abs() + 1e-6
    assert bool((err <= tol).all()), f"max err {err.max().item()}"


@pytest.mark.parametrize("R,N,K", [(1, 256, 64), (5, 200, 136), (32, 7168, 7168), (17, 1000, 2064),
                                   (32, 18432, 7168), (3, 300, 18432)])
def test_decode_gemm(R, N, K):
    """The draft step's bf16 decode GEMM (weights on the N = 256 side, stream-K
    ranges, atomics across CTAs): out += x W^T against the fp32 product of the
    same bf16 values; ragged N and K, 1..32 tokens."""
    g = torch.Generator(device="cuda").manual_seed(R + N + K)
    x = torch.randn(R, K, device="cuda", generator=g).to(torch.bfloat16)
    w = (0.05 * torch.randn(N, K, device="cuda", generator=g)).to(torch.bfloat16)
    out0 = torch.randn(R, N, device="cuda", generator=g)
    out = out0.clone()
    lib.gemm_decode_bf16(x, w, out)
    lib.check_errors()
    ref = out0.double() + x.double() @ w.double().T
    err = (out.double() - ref).abs()
    tol = 1e-5 * (x.double().abs() @ w.double().abs().T) + 1e-5 * out0.double().abs() + 1e-6
    assert bool((err <= tol).all()), f"max err {err.max().item()}"
