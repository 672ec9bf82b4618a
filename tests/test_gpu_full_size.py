"""Parity at the full workload sizes, in the launch configuration bench.py
times, on outputs the oracle can compute one by one: sampled rows of y and
dX, sampled neurons of dWg / dWu / dWd, plus properties that hold at any size
(routing consistency, counts).  Tolerance as in test_gpu_ffn.py, with the
gate-decision allowance computed from the oracle for the sampled outputs."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from activation_sparse_gated_tcgen05_gb300 import synthetic, twell

from helpers import (assert_close, bwd_allowance_sampled, dev_bf16, fwd_allowance,
                     to_np)

pytestmark = pytest.mark.gpu
LAM = 2e-5


@pytest.fixture(scope="module", autouse=True)
def _oracle_threads():
    oracle.set_threads(os.cpu_count() or 1)
    yield
    oracle.set_threads(1)


def _sample(n, k, seed):
    rng = np.random.default_rng(seed)
    pick = rng.choice(n, size=min(k, n), replace=False)
    return np.unique(np.concatenate([[0, n - 1], pick])).astype(np.int64)


def _upload(w, keys):
    return [dev_bf16(w[k]) for k in keys]


def _check_route(tiles, route, shape, W):
    M = shape.M
    _, _, cnt, nnz = twell.tiles_view(tiles, shape)
    cnt, nnz = cnt.cpu().numpy(), nnz.cpu().numpy()
    ev, ec, en, dr, nd = twell.hybrid_view(route, shape)
    n = int(nd.item())
    dr = dr[:n].cpu().numpy()
    en = en.cpu().numpy()
    routed = np.zeros(M, bool)
    routed[dr] = True
    assert (np.diff(dr) > 0).all()                       # ascending, unique
    want = (cnt > shape.tile_cap).any(1) | (nnz > W)
    np.testing.assert_array_equal(routed, want)
    np.testing.assert_array_equal(en[~routed], nnz[~routed])
    assert not en[routed].any()
    assert int(cnt.astype(np.int64).sum()) == int(nnz.sum())
    return n


def _fwd_inference(w, wl, M=None):
    """The TwELL forward as bench.py runs it: with the optional workspace,
    which for d_model > 1024 selects the split up / down gathers.  Where it
    does, the forward without a workspace (the fused gather) must give the
    same bytes."""
    M = wl.M if M is None else M
    x, wg, wu, wd = _upload(w, ("x", "wgT", "wuT", "wd"))
    shape = twell.make_shape(M, wl.d_model, wl.d_ff, wl.tile_n, wl.tile_cap)
    tiles = twell.alloc_tiles(shape)
    twell.twell_pack(x, wg, shape, tiles)
    y = torch.empty(M, wl.d_model, dtype=torch.bfloat16, device="cuda")
    nbytes = twell.twell_tiles_workspace_bytes(shape)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if nbytes else None
    twell.twell_ffn_fwd(x, wg, wu, wd, shape, y, tiles=tiles, ws=ws)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 0
    if ws is not None:
        y_fused = torch.empty_like(y)
        twell.twell_ffn_fwd(x, wg, wu, wd, shape, y_fused, tiles=tiles)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y_fused.view(torch.int16))
    return y, tiles, shape


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_fwd_0p5b_forward(seed):
    wl = synthetic.WORKLOADS["fwd_0p5b"]
    w = synthetic.make_workload(wl, seed=seed, with_dy=False)
    y, tiles, shape = _fwd_inference(w, wl)
    nnz = twell.tiles_view(tiles, shape)[3].cpu().numpy()
    assert abs(nnz.mean() / wl.d_ff - wl.density) < 0.05 * wl.density
    rows = _sample(wl.M, 24, seed)
    ref = oracle.ffn_fwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"], rows=rows)
    assert_close(to_np(y)[rows], ref, "y", out_bf16=True, allowance=fwd_allowance(w, rows))


@pytest.mark.parametrize("density", synthetic.DENSITY_SWEEP)
def test_fwd_2b_density_sweep_forward(density):
    wl = synthetic.WORKLOADS["fwd_2b"]
    w = synthetic.make_workload(wl, density=density, with_dy=False)
    y, tiles, shape = _fwd_inference(w, wl)
    rows = _sample(wl.M, 12, 3)
    ref = oracle.ffn_fwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"], rows=rows)
    assert_close(to_np(y)[rows], ref, "y", out_bf16=True, allowance=fwd_allowance(w, rows))


def _pass_boundaries(f, d):
    """First neurons of the L2-sized neuron passes of the wide-row gathers
    (one weight matrix per pass for the up / down / dh / gradient gathers,
    two for dX), by the library's rule: one pass while the table fits in
    3/4 of L2, else passes of at most half of L2 each."""
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    out = set()
    for table in (2.0 * f * d, 4.0 * f * d):
        n = 1 if table <= 0.75 * l2 else math.ceil(table / (0.5 * l2))
        out.update(f * c // n for c in range(1, n))
    return sorted(out)


@pytest.mark.parametrize("name", ["train_2b", "train_8b"])
def test_training_step(name):
    wl = synthetic.WORKLOADS[name]
    w = synthetic.make_workload(wl)
    M, d, f = wl.M, wl.d_model, wl.d_ff
    x, wg, wu, wd, dy = _upload(w, ("x", "wgT", "wuT", "wd", "dy"))
    shape = twell.make_shape(M, d, f, wl.tile_n, wl.tile_cap)
    tiles = twell.alloc_tiles(shape)
    twell.twell_pack(x, wg, shape, tiles)
    nnz = twell.tiles_view(tiles, shape)[3].cpu().numpy()
    W = synthetic.ell_width(nnz, wl.route_fraction)
    route = twell.alloc_hybrid(shape, W)
    twell.hybrid_route(tiles, shape, route)
    # as bench.py runs it: a workspace for exactly the rows routed
    route.dense_cap = int(route.n_dense[0].item())
    ws = torch.empty(twell.twell_workspace_bytes(shape, W, True, dense_cap=route.dense_cap),
                     dtype=torch.uint8, device="cuda")
    y = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    twell.twell_ffn_fwd(x, wg, wu, wd, shape, y, route=route, ws=ws)
    dx = torch.empty_like(y)
    dws = [torch.full((f, d), float("nan"), device="cuda") for _ in range(3)]
    twell.twell_ffn_bwd(x, wg, wu, wd, dy, shape, route, LAM, dx, *dws, ws)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 0
    n_dense = _check_route(tiles, route, shape, W)
    assert 0.01 * M < n_dense < 0.06 * M  # about 3 % of rows routed
    dr = twell.hybrid_view(route, shape)[3][:n_dense].cpu().numpy()
    rng = np.random.default_rng(5)
    # rows: random ones, the last rows (the final row block of every gather
    # pass), and among the routed rows the first and the last row of every
    # 128-row tile of the dense backup's buffer
    tile_rows = [dr[i] for k in range(0, n_dense, 128) for i in (k, min(k + 127, n_dense - 1))]
    rows = np.unique(np.concatenate([_sample(M, 8, 4), [M - 2, M - 3],
                                     rng.choice(dr, 2, replace=False), tile_rows]))
    # neurons: random ones and both sides of every L2-pass boundary
    edges = [j + o for j in _pass_boundaries(f, d) for o in (-1, 0)]
    neurons = np.unique(np.concatenate([_sample(f, 6, 6), edges])).astype(np.int64)
    y_ref = oracle.ffn_fwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"], rows=rows)
    assert_close(to_np(y)[rows], y_ref, "y", out_bf16=True, allowance=fwd_allowance(w, rows))
    al = bwd_allowance_sampled(w, LAM, rows, neurons)
    dx_ref = oracle.ffn_bwd_dx_rows(w["x"], w["wgT"], w["wuT"], w["wd"], w["dy"], LAM, rows)
    assert_close(to_np(dx)[rows], dx_ref, "dx", out_bf16=True, allowance=al["dx"])
    og, ou, od = oracle.ffn_bwd_dw_neurons(w["x"], w["wgT"], w["wuT"], w["wd"], w["dy"], LAM,
                                           neurons)
    assert_close(dws[0].cpu().numpy()[neurons], og, "dwgT", allowance=al["dwgT"])
    assert_close(dws[1].cpu().numpy()[neurons], ou, "dwuT", allowance=al["dwuT"])
    assert_close(dws[2].cpu().numpy()[neurons], od, "dwd", allowance=al["dwd"])


def test_train_8b_small_batch_forward():
    wl = synthetic.WORKLOADS["train_8b"]
    w = synthetic.make_workload(wl, M=64, with_dy=False)
    for M in sorted(set(synthetic.SMALL_M) | {3}):
        sub = {k: (v[:M] if k == "x" else v) for k, v in w.items() if k != "row_density"}
        y, _, _ = _fwd_inference(sub, wl, M=M)
        ref = oracle.ffn_fwd_dense(sub["x"], sub["wgT"], sub["wuT"], sub["wd"])
        assert_close(to_np(y), ref, "y M=%d" % M, out_bf16=True, allowance=fwd_allowance(sub))
