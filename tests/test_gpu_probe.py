"""The benchmark's row-gather probe (libtwell_probe.so): it reads the rows it
is given, skips ids outside the table and rejects an output buffer smaller
than one word per warp."""
import numpy as np
import pytest
import torch

from activation_sparse_gated_tcgen05_gb300 import probe

pytestmark = pytest.mark.gpu


def _fold(table, idx, rows, warps):
    t = table.cpu().numpy().view(np.uint32).reshape(rows, -1)
    i = idx.cpu().numpy()
    out = []
    for w in range(warps):
        ids = i[w::warps]
        ids = ids[(ids >= 0) & (ids < rows)]
        out.append(np.bitwise_xor.reduce(t[ids].reshape(-1)) if ids.size else np.uint32(0))
    return np.array(out, np.uint32)


def test_gather_probe_reads_rows():
    rows, row_bytes = 1024, 2048
    table = torch.randint(0, 2 ** 31 - 1, (rows * row_bytes // 4,), dtype=torch.int32).cuda()
    idx = torch.randint(0, rows, (4096,), dtype=torch.int32).cuda()
    out = torch.zeros(8 * 4, dtype=torch.int32).cuda()
    probe.gather(table, row_bytes, idx, out, 4)
    torch.cuda.synchronize()
    # warp w reads rows idx[w], idx[w + 32], ...
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), _fold(table, idx, rows, 32))


def test_gather_probe_skips_ids_outside_the_table():
    rows, row_bytes = 64, 512
    table = torch.randint(0, 2 ** 31 - 1, (rows * row_bytes // 4,), dtype=torch.int32).cuda()
    idx = torch.tensor([3, -1, rows, 5, rows + 100, 63, 0, -7] * 16, dtype=torch.int32).cuda()
    out = torch.zeros(8 * 2, dtype=torch.int32).cuda()
    probe.gather(table, row_bytes, idx, out, 2)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), _fold(table, idx, rows, 16))


def test_gather_probe_rejects_a_short_output():
    table = torch.zeros(1024, dtype=torch.int32).cuda()
    idx = torch.zeros(16, dtype=torch.int32).cuda()
    out = torch.zeros(8 * 4 - 1, dtype=torch.int32).cuda()
    with pytest.raises(RuntimeError):
        probe.gather(table, 256, idx, out, 4)
