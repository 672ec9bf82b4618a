"""Failure detection without a GPU fault: a device-side wait that nothing
completes gives up after its limit, records TWELL_ERR_DEVICE_TIMEOUT in the
status word, and leaves the context usable for the next call."""
import time

import numpy as np
import pytest
import torch

from activation_sparse_gated_tcgen05_gb300 import twell

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    assert twell.twell_get_device_status() == 0
    t0 = time.time()
    twell.twell_selftest_wait_timeout(50_000)  # 50 ms
    assert twell.twell_get_device_status() == 6  # TWELL_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 10.0
    assert twell.twell_get_device_status() == 0  # cleared by the read
    # the context still works: a small exact GEMM through the same library
    A = torch.randint(-2, 3, (128, 64)).to(torch.bfloat16).cuda()
    B = torch.randint(-2, 3, (256, 64)).to(torch.bfloat16).cuda()
    C = torch.empty(128, 256, dtype=torch.float32, device="cuda")
    twell.twell_gemm_bf16(A, B, C, 128, 256, 64, False, False)
    torch.cuda.synchronize()
    ref = A.double().cpu() @ B.double().cpu().t()
    np.testing.assert_array_equal(C.cpu().double().numpy(), ref.numpy())

