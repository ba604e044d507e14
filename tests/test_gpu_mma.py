"""Tensor-core building block: one tcgen05.mma tile from 128-byte-swizzled
shared memory (K-major and MN-major operands; TF32 MN-major operands in the
128-byte swizzle of 32-byte atoms), checked against a CPU product."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _tf32_trunc(x):
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) & np.uint32(0xFFFFE000)
    return u.view(np.float32)


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("M,N", [(128, 32), (128, 64), (128, 128), (128, 256), (64, 32),
                                 (64, 128)])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)])
def test_single_tile_product(dtype, M, N, a_mn, b_mn):
    W_ = 32 if dtype == 0 else 64
    if (a_mn and M % W_) or (b_mn and N % W_):
        pytest.skip("an MN-major operand spans whole 128-byte blocks")
    import torch
    import attention_backward_pass_gb300 as ab
    W = 32 if dtype == 0 else 64
    K = 2 * W
    rng = np.random.default_rng(M * 1000 + N + 10 * a_mn + b_mn)
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((N, K)).astype(np.float32)
    if dtype == 1:
        tA = torch.from_numpy(A).to(torch.bfloat16)
        tB = torch.from_numpy(B).to(torch.bfloat16)
        A64 = tA.float().numpy().astype(np.float64)
        B64 = tB.float().numpy().astype(np.float64)
    else:
        tA, tB = torch.from_numpy(A), torch.from_numpy(B)
        A64, B64 = _tf32_trunc(A).astype(np.float64), _tf32_trunc(B).astype(np.float64)
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    ab.selftest_mma(dtype, M, N, K, a_mn, b_mn, tA.cuda(), tB.cuda(), C)
    torch.cuda.synchronize()
    ref = A64 @ B64.T
    err = np.max(np.abs(C.cpu().numpy() - ref)) / np.max(np.abs(ref))
    # inputs are exactly representable in the operand type; only the fp32
    # accumulation order differs (and TF32 rounding of fp32 inputs)
    assert err < (2e-3 if dtype == 0 else 1e-5), err


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("M,N", [(128, 32), (128, 64), (128, 128), (64, 32), (64, 64)])
@pytest.mark.parametrize("b_mn", [0, 1])
def test_a_operand_from_tmem(dtype, M, N, b_mn):
    W_ = 32 if dtype == 0 else 64
    if b_mn and N % W_:
        pytest.skip("an MN-major operand spans whole 128-byte blocks")
    import torch
    import attention_backward_pass_gb300 as ab
    K = 2 * W_
    rng = np.random.default_rng(7 + M + N)
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((N, K)).astype(np.float32)
    if dtype == 1:
        tA = torch.from_numpy(A).to(torch.bfloat16)
        tB = torch.from_numpy(B).to(torch.bfloat16)
        A64 = tA.float().numpy().astype(np.float64)
        B64 = tB.float().numpy().astype(np.float64)
    else:
        tA, tB = torch.from_numpy(A), torch.from_numpy(B)
        A64, B64 = _tf32_trunc(A).astype(np.float64), _tf32_trunc(B).astype(np.float64)
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    ab.selftest_mma(dtype, M, N, K, 0, b_mn, tA.cuda(), tB.cuda(), C, a_tmem=True)
    torch.cuda.synchronize()
    ref = A64 @ B64.T
    err = np.max(np.abs(C.cpu().numpy() - ref)) / np.max(np.abs(ref))
    assert err < (2e-3 if dtype == 0 else 1e-5), err
