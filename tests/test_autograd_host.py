"""Host logic of the autograd binding (no GPU): the ELL-width policy."""
import torch

from activation_sparse_gated_tcgen05_gb300.autograd import ell_width_for


def test_ell_width_widest_row_when_nothing_routed():
    nnz = torch.tensor([3, 9, 1, 7], dtype=torch.int32)
    assert ell_width_for(nnz, 0.0) == 9


def test_ell_width_quantile_routes_the_fraction():
    nnz = torch.arange(100, dtype=torch.int32).flip(0)  # 99 .. 0
    W = ell_width_for(nnz, 0.03)
    assert W == 97                         # sorted index floor(0.97 * 100)
    assert int((nnz > W).sum()) == 2       # rows above W go to the dense fallback


def test_ell_width_empty_batch():
    assert ell_width_for(torch.zeros(0, dtype=torch.int32), 0.03) == 0
