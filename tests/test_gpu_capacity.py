"""Routed-row capacity of the hybrid path (twell_hybrid.dense_cap) and the
memory a training step takes with it.

A workspace sized for exactly the rows routed gives the same bytes as one
sized for every row; routing more rows than the capacity records
TWELL_ERR_CAPACITY without a fault; and a sparse training step, buffers
included, takes less device memory than the library's dense one (page 2,
"¿Cuánto se acelera realmente?", reports lower peak memory for the sparse
model)."""
import numpy as np
import pytest
import torch

from activation_sparse_gated_tcgen05_gb300 import synthetic, twell

from helpers import dev_bf16

pytestmark = pytest.mark.gpu
LAM = 2e-5


def _inputs(M, d, f, tile_n, cap, exact=True, seed=3, mixed=True):
    if exact:
        w = synthetic.make_exact_gate_inputs(M, d, f, density=0.02, seed=seed, mixed_rows=mixed)
    else:
        w = synthetic.make_inputs(M, d, f, density=0.005, seed=seed, lognormal_sigma=1.0)
    x, wg, wu, wd, dy = (dev_bf16(w[k]) for k in ("x", "wgT", "wuT", "wd", "dy"))
    return x, wg, wu, wd, dy, twell.make_shape(M, d, f, tile_n, cap)


def _step(x, wg, wu, wd, dy, shape, W, dense_cap):
    """pack, route, forward, backward with a workspace for dense_cap routed rows."""
    M, d, f = shape.M, shape.d_model, shape.d_ff
    tiles = twell.alloc_tiles(shape)
    twell.twell_pack(x, wg, shape, tiles)
    route = twell.alloc_hybrid(shape, W, dense_cap=dense_cap)
    twell.hybrid_route(tiles, shape, route)
    nbytes = twell.twell_workspace_bytes(shape, W, True, dense_cap=dense_cap)
    ws = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
    y = torch.full((M, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    twell.twell_ffn_fwd(x, wg, wu, wd, shape, y, route=route, ws=ws)
    dx = torch.full_like(y, float("nan"))
    dws = [torch.full((f, d), float("nan"), device="cuda") for _ in range(3)]
    twell.twell_ffn_bwd(x, wg, wu, wd, dy, shape, route, LAM, dx, *dws, ws)
    torch.cuda.synchronize()
    return y, dx, dws, int(route.n_dense[0].item()), nbytes


def _same(a, b):
    return torch.equal(a.contiguous().view(torch.int16 if a.element_size() == 2 else torch.int32),
                       b.contiguous().view(torch.int16 if b.element_size() == 2 else torch.int32))


@pytest.mark.parametrize("M,d,f,tile_n,cap,q", [(300, 256, 1024, 64, 16, 0.9),
                                                (700, 2048, 1024, 128, 32, 0.7),
                                                (1000, 1024, 2048, 128, 32, 1.0)])
def test_capped_workspace_gives_the_same_bytes(M, d, f, tile_n, cap, q):
    x, wg, wu, wd, dy, shape = _inputs(M, d, f, tile_n, cap)
    t = twell.alloc_tiles(shape)
    twell.twell_pack(x, wg, shape, t)
    nnz = twell.tiles_view(t, shape)[3].cpu().numpy()
    W = int(np.sort(nnz)[int(q * (M - 1))])
    y0, dx0, dw0, n0, b0 = _step(x, wg, wu, wd, dy, shape, W, M)
    assert twell.twell_get_device_status() == 0
    y1, dx1, dw1, n1, b1 = _step(x, wg, wu, wd, dy, shape, W, n0)
    assert twell.twell_get_device_status() == 0
    assert n1 == n0
    if n0 < M - 128:
        assert b1 < b0  # the dense-backup buffers shrink with the capacity
    assert _same(y0, y1) and _same(dx0, dx1)
    for a, b in zip(dw0, dw1):
        assert _same(a, b)


def test_zero_capacity_without_routed_rows():
    # the widest row as ELL width and capacity zero: no dense-backup launch
    M, d, f = 512, 512, 1024
    x, wg, wu, wd, dy, shape = _inputs(M, d, f, 128, 32, mixed=False)
    t = twell.alloc_tiles(shape)
    twell.twell_pack(x, wg, shape, t)
    _, _, cnt, nnz = twell.tiles_view(t, shape)
    assert int(cnt.max().item()) <= 32  # no tile overflows at this density
    W = int(nnz.max().item())
    y0, dx0, dw0, n0, _ = _step(x, wg, wu, wd, dy, shape, W, M)
    assert n0 == 0
    launches = twell.twell_launch_count()
    y1, dx1, dw1, _, _ = _step(x, wg, wu, wd, dy, shape, W, 0)
    fewer = twell.twell_launch_count() - launches
    launches = twell.twell_launch_count()
    _step(x, wg, wu, wd, dy, shape, W, M)
    full = twell.twell_launch_count() - launches
    assert fewer < full
    assert twell.twell_get_device_status() == 0
    assert _same(y0, y1) and _same(dx0, dx1)
    for a, b in zip(dw0, dw1):
        assert _same(a, b)


def test_routing_past_the_capacity_reports_capacity():
    M, d, f = 300, 256, 1024
    x, wg, wu, wd, dy, shape = _inputs(M, d, f, 64, 16)
    t = twell.alloc_tiles(shape)
    twell.twell_pack(x, wg, shape, t)
    nnz = twell.tiles_view(t, shape)[3].cpu().numpy()
    W = int(np.sort(nnz)[int(0.5 * (M - 1))])
    route = twell.alloc_hybrid(shape, W)
    twell.hybrid_route(t, shape, route)
    n = int(route.n_dense[0].item())
    assert n > 2
    assert twell.twell_get_device_status() == 0
    for cap in (n - 1, n // 3, 0):
        _step(x, wg, wu, wd, dy, shape, W, cap)  # runs to the end, no fault
        assert twell.twell_get_device_status() == 4  # TWELL_ERR_CAPACITY
        assert twell.twell_get_device_status() == 0  # read clears it
    _step(x, wg, wu, wd, dy, shape, W, n)
    assert twell.twell_get_device_status() == 0


def test_sparse_training_step_takes_less_memory_than_dense():
    # a mid-size training shape with lognormal row densities (median 0.5 %),
    # 3 % of the rows routed: every buffer of the step is allocated inside
    # the measured window, from a state holding only inputs and weights
    M, d, f = 4096, 1024, 4096
    x, wg, wu, wd, dy, shape = _inputs(M, d, f, 128, 32, exact=False)
    t = twell.alloc_tiles(shape)
    twell.twell_pack(x, wg, shape, t)
    W = synthetic.ell_width(twell.tiles_view(t, shape)[3].cpu().numpy(), 0.03)
    del t

    def peak(run):
        torch.cuda.synchronize()
        base = torch.cuda.memory_allocated()
        torch.cuda.reset_peak_memory_stats()
        run()
        torch.cuda.synchronize()
        return torch.cuda.max_memory_allocated() - base

    def sparse():
        tiles = twell.alloc_tiles(shape)
        twell.twell_pack(x, wg, shape, tiles)
        route = twell.alloc_hybrid(shape, W)
        twell.hybrid_route(tiles, shape, route)
        del tiles
        route.dense_cap = int(route.n_dense[0].item())
        assert 0 < route.dense_cap < 0.06 * M
        ws = torch.empty(twell.twell_workspace_bytes(shape, W, True, dense_cap=route.dense_cap),
                         dtype=torch.uint8, device="cuda")
        y = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
        twell.twell_ffn_fwd(x, wg, wu, wd, shape, y, route=route, ws=ws)
        dx = torch.empty_like(y)
        dws = [torch.empty(f, d, device="cuda") for _ in range(3)]
        twell.twell_ffn_bwd(x, wg, wu, wd, dy, shape, route, LAM, dx, *dws, ws)

    def dense():
        ws = torch.empty(twell.twell_dense_workspace_bytes(shape, True), dtype=torch.uint8,
                         device="cuda")
        y = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
        twell.twell_dense_ffn_fwd(x, wg, wu, wd, shape, y, True, ws)
        dx = torch.empty_like(y)
        dws = [torch.empty(f, d, device="cuda") for _ in range(3)]
        twell.twell_dense_ffn_bwd(x, wg, wu, wd, dy, shape, LAM, dx, *dws, ws)

    sp, de = peak(sparse), peak(dense)
    assert twell.twell_get_device_status() == 0
    outputs = 2 * M * d * 2 + 3 * f * d * 4  # y, dX, dW: the same for both
    assert sp < de
    # beyond the outputs both need, the sparse step's own buffers are well
    # under half of the dense step's (which keeps g, u, h and du, da)
    assert sp - outputs < 0.5 * (de - outputs), (sp, de, outputs)
