"""tcgen05 GEMM engine through the C ABI (twell_gemm_bf16): all four operand
majorness combinations, ragged tails, bf16 / fp32 outputs and accumulation,
each in both GEMM forms (CTA-pair 256 x 256 tiles and single-CTA 128 x 256
tiles, twell_set_pair_gemm).

Integer-valued operands make every product and partial sum exact in fp32, so
those cases must match bit for bit; random operands are checked against a
float64 CPU matmul."""
import numpy as np
import pytest
import torch

from activation_sparse_gated_tcgen05_gb300 import twell

from helpers import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[True, False], ids=["pair", "single"], autouse=True)
def gemm_form(request):
    """Every case runs with CTA-pair tiles (the default) and single-CTA tiles."""
    prev = twell.twell_set_pair_gemm(request.param)
    yield request.param
    twell.twell_set_pair_gemm(prev)


def _operands(M, N, K, a_mn, b_mn, integer, seed):
    g = torch.Generator().manual_seed(seed)
    if integer:
        A = torch.randint(-3, 4, (M, K), generator=g).double()
        B = torch.randint(-3, 4, (N, K), generator=g).double()
    else:
        A = torch.randn(M, K, generator=g, dtype=torch.float64)
        B = torch.randn(N, K, generator=g, dtype=torch.float64)
    A = A.to(torch.bfloat16).double()
    B = B.to(torch.bfloat16).double()
    a_store = (A.t() if a_mn else A).contiguous().to(torch.bfloat16).cuda()
    b_store = (B.t() if b_mn else B).contiguous().to(torch.bfloat16).cuda()
    return A, B, a_store, b_store


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 264, 72), (1000, 520, 328)])
def test_gemm_integer_exact(a_mn, b_mn, M, N, K):
    if a_mn and M % 8:
        pytest.skip("MN-major A needs M % 8 == 0")
    A, B, a, b = _operands(M, N, K, a_mn, b_mn, True, 1)
    C = torch.empty(M, N, dtype=torch.float32, device="cuda")
    twell.twell_gemm_bf16(a, b, C, M, N, K, a_mn, b_mn)
    torch.cuda.synchronize()
    ref = (A @ B.t()).numpy()
    np.testing.assert_array_equal(C.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_gemm_random_bf16_out_and_accumulate(a_mn, b_mn):
    M, N, K = 1040, 776, 1096
    A, B, a, b = _operands(M, N, K, a_mn, b_mn, False, 2)
    ref = (A @ B.t()).numpy()
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    twell.twell_gemm_bf16(a, b, C, M, N, K, a_mn, b_mn)
    torch.cuda.synchronize()
    assert_close(C.float().cpu().numpy(), ref, "bf16 out", out_bf16=True)
    C32 = torch.full((M, N), 0.5, dtype=torch.float32, device="cuda")
    twell.twell_gemm_bf16(a, b, C32, M, N, K, a_mn, b_mn, accumulate=True)
    torch.cuda.synchronize()
    assert_close(C32.cpu().numpy(), ref + 0.5, "fp32 accumulate", rel=1e-5, max_rms=1e-4)


def test_gemm_many_tiles_persistent_wraparound():
    # more tiles than SMs so every CTA loops over several tiles and both
    # TMEM accumulators and all smem stages wrap around
    M, N, K = 4096, 4096, 512
    A, B, a, b = _operands(M, N, K, 0, 0, True, 3)
    C = torch.empty(M, N, dtype=torch.float32, device="cuda")
    twell.twell_gemm_bf16(a, b, C, M, N, K, 0, 0)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 0
    ref = (A.cuda() @ B.cuda().t()).cpu().numpy()  # exact integers in fp64
    np.testing.assert_array_equal(C.cpu().numpy().astype(np.float64), ref)


def test_pair_and_single_forms_agree_bit_for_bit():
    # random bf16 operands: both forms accumulate the same products over K in
    # the same order, so their fp32 outputs are identical
    M, N, K = 2048, 1536, 1024
    _, _, a, b = _operands(M, N, K, 0, 1, False, 4)
    out = {}
    for pair in (True, False):
        prev = twell.twell_set_pair_gemm(pair)
        C = torch.empty(M, N, dtype=torch.float32, device="cuda")
        twell.twell_gemm_bf16(a, b, C, M, N, K, 0, 1)
        torch.cuda.synchronize()
        twell.twell_set_pair_gemm(prev)
        out[pair] = C
    assert twell.twell_get_device_status() == 0
    assert torch.equal(out[True].view(torch.int32), out[False].view(torch.int32))
