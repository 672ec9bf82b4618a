"""The allocation-free hybrid forward (twell_ffn_fwd_noalloc) gives the same
result as twell_ffn_fwd with a caller workspace, on two calls in a row.

It is for callers that cannot allocate device memory when they run the FFN
(stream capture, a host runtime that owns allocation, a fixed memory budget);
its scratch is a fixed array inside the library.  This file is collected last
so a failure here leaves every other test already run."""
import numpy as np
import pytest
import torch

from activation_sparse_gated_tcgen05_gb300 import synthetic, twell

from helpers import assert_close, dev_bf16, to_np

pytestmark = pytest.mark.gpu


def _setup(M, d, f, tile_n, cap, q):
    w = synthetic.make_exact_gate_inputs(M, d, f, density=0.02, seed=7, mixed_rows=True)
    x, wg, wu, wd = (dev_bf16(w[k]) for k in ("x", "wgT", "wuT", "wd"))
    shape = twell.make_shape(M, d, f, tile_n, cap)
    tiles = twell.alloc_tiles(shape)
    twell.twell_pack(x, wg, shape, tiles)
    nnz = twell.tiles_view(tiles, shape)[3].cpu().numpy()
    W = int(np.sort(nnz)[int(q * (M - 1))])
    route = twell.alloc_hybrid(shape, W)
    twell.hybrid_route(tiles, shape, route)
    return x, wg, wu, wd, shape, route, W


@pytest.mark.parametrize("M,d,f,tile_n,cap", [(300, 256, 1024, 64, 16), (1024, 1024, 4096, 128, 32),
                                              (256, 2048, 1024, 128, 32)])
def test_noalloc_forward_matches_workspace_forward(M, d, f, tile_n, cap):
    x, wg, wu, wd, shape, route, W = _setup(M, d, f, tile_n, cap, 0.8)
    assert twell.twell_workspace_bytes(shape, W, False) <= 32 << 20
    ws = torch.empty(twell.twell_workspace_bytes(shape, W, False), dtype=torch.uint8, device="cuda")
    y_ref = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    twell.twell_ffn_fwd(x, wg, wu, wd, shape, y_ref, route=route, ws=ws)
    assert int(route.n_dense[0].item()) > 0  # the scratch path is really used
    for _ in range(2):
        y = torch.full((M, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        twell.twell_ffn_fwd_noalloc(x, wg, wu, wd, shape, y, route)
        torch.cuda.synchronize()
        assert_close(to_np(y), to_np(y_ref), "y", out_bf16=True)
        # the same kernels on the same inputs: the scratch only moves buffers
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    assert twell.twell_get_device_status() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    M, d, f = 8192, 1024, 4096
    shape = twell.make_shape(M, d, f, 128, 32)
    assert twell.twell_workspace_bytes(shape, 32, False) > 32 << 20
    x = torch.zeros(M, d, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(f, d, dtype=torch.bfloat16, device="cuda")
    route = twell.alloc_hybrid(shape, 32)
    y = torch.empty_like(x)
    with pytest.raises(twell.TwellError) as e:
        twell.twell_ffn_fwd_noalloc(x, w, w, w, shape, y, route)
    assert e.value.status == 7  # TWELL_ERR_WORKSPACE
