"""The ELL forward gather split into L2-sized neuron passes.

When the gathered weight rows exceed about 3/4 of L2, the gathers of page 2
"Sakana AI and NVIDIA introduce TwELL with CUDA kernels ...", section "¿Qué
hace distinto a TwELL frente a ELL clásico?" run once per neuron chunk and
carry y_m between passes in fp32.  Up to d_model = 1024 the fused up+down
kernel gathers Wu^T and Wd rows together (4 * d_ff * d_model bytes); wider
rows split it into an up gather (Wu^T) and a down gather (Wd), each with its
own passes over 2 * d_ff * d_model bytes.  A row's ELL columns ascend, every
chunk is a contiguous slice of it and the per-entry arithmetic and
accumulation order are unchanged, so the result must equal the single-pass
fused TwELL forward bit for bit; sampled rows are also checked against the
oracle."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from activation_sparse_gated_tcgen05_gb300 import synthetic, twell

from helpers import assert_close, dev_bf16, fwd_allowance, to_np

pytestmark = pytest.mark.gpu


def _expected_passes(table_bytes):
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    return 1 if table_bytes <= 0.75 * l2 else math.ceil(table_bytes / (0.5 * l2))


# M large enough that the TwELL forward runs one team per row (batches of
# fewer than two row groups per SM split rows over clusters, which sums in
# another order): eight rows per group at d = 1024, two at d = 2048 and 4096.
# d_ff is chosen so that the gathered table exceeds L2: the fused kernel's
# Wu^T + Wd at d = 1024, Wu^T or Wd alone for the split gathers.
@pytest.mark.parametrize("rows_per_group,d,f", [(8, 1024, 32768), (2, 2048, 32768),
                                                (2, 4096, 16384)])
def test_multi_pass_forward_matches_single_pass(rows_per_group, d, f):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M = 2 * sms * rows_per_group + 37
    split = d > 1024
    passes = _expected_passes((2.0 if split else 4.0) * f * d)
    assert passes > 1, "shape no longer exceeds L2; pick a larger one"
    w = synthetic.make_inputs(M, d, f, seed=11, with_dy=False)
    x, wg, wu, wd = (dev_bf16(w[k]) for k in ("x", "wgT", "wuT", "wd"))
    shape = twell.make_shape(M, d, f, 128, 32)
    tiles = twell.alloc_tiles(shape)
    twell.twell_pack(x, wg, shape, tiles)
    nnz = twell.tiles_view(tiles, shape)[3].cpu().numpy()
    W = int(nnz.max())  # no row routed: every row goes through the gather
    route = twell.alloc_hybrid(shape, W)
    twell.hybrid_route(tiles, shape, route)
    ws = torch.empty(twell.twell_workspace_bytes(shape, W, False), dtype=torch.uint8,
                     device="cuda")
    y_single = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    twell.twell_ffn_fwd(x, wg, wu, wd, shape, y_single, tiles=tiles)
    y_multi = torch.full((M, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    twell.twell_profile_begin("*")
    twell.twell_ffn_fwd(x, wg, wu, wd, shape, y_multi, route=route, ws=ws)
    torch.cuda.synchronize()
    prof = twell.twell_profile_end()
    assert twell.twell_get_device_status() == 0
    assert int(twell.hybrid_view(route, shape)[4].item()) == 0
    families = ("sparse_fwd_up", "sparse_fwd_down") if split else ("sparse_fwd",)
    for fam in families:
        assert prof[fam][0] == passes, (fam, prof)
    if split:
        assert "sparse_fwd" not in prof
    # same bytes: entries in the same order, fp32 carried exactly between passes
    assert torch.equal(y_multi.view(torch.int16), y_single.view(torch.int16))
    rows = np.array([0, 1, M // 2, M - 1], dtype=np.int64)
    oracle.set_threads(os.cpu_count() or 1)
    try:
        ref = oracle.ffn_fwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"], rows=rows)
    finally:
        oracle.set_threads(1)
    assert_close(to_np(y_multi)[rows], ref, "y", out_bf16=True, allowance=fwd_allowance(w, rows))


def _chunks(table_bytes, fit, chunk):
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    return 1 if table_bytes <= fit * l2 else math.ceil(table_bytes / (chunk * l2))


@pytest.mark.parametrize("d,f", [(1024, 16384), (4096, 16384)])
def test_multi_pass_backward_rows(d, f):
    """dX over ELL rows in L2-sized passes: sampled rows of dX and sampled
    neurons of the weight gradients against the oracle, and the pass counts
    seen by the profiler.  Up to d_model = 1024 the fused row kernel gathers
    Wd, Wu^T and Wg^T together; wider rows split it into dh (Wd) and u, the
    gradients and dX (Wu^T and Wg^T), each with its own passes."""
    from helpers import bwd_allowance_sampled

    M, lam = 256, 2e-5
    if d <= 1024:
        expect = {"bwd_rows": _chunks(6.0 * f * d, 0.5, 0.65)}
    else:
        expect = {"bwd_dh": _chunks(2.0 * f * d, 0.75, 0.5),
                  "bwd_grad_dx": _chunks(4.0 * f * d, 0.75, 0.5)}
    assert min(expect.values()) > 1, "shape no longer exceeds L2; pick a larger one"
    w = synthetic.make_inputs(M, d, f, seed=12)
    x, wg, wu, wd, dy = (dev_bf16(w[k]) for k in ("x", "wgT", "wuT", "wd", "dy"))
    shape = twell.make_shape(M, d, f, 128, 32)
    tiles = twell.alloc_tiles(shape)
    twell.twell_pack(x, wg, shape, tiles)
    W = int(twell.tiles_view(tiles, shape)[3].max().item())
    route = twell.alloc_hybrid(shape, W)
    twell.hybrid_route(tiles, shape, route)
    ws = torch.empty(twell.twell_workspace_bytes(shape, W, True), dtype=torch.uint8,
                     device="cuda")
    dx = torch.full((M, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    dws = [torch.full((f, d), float("nan"), device="cuda") for _ in range(3)]
    twell.twell_profile_begin("*")
    twell.twell_ffn_bwd(x, wg, wu, wd, dy, shape, route, lam, dx, *dws, ws)
    torch.cuda.synchronize()
    prof = twell.twell_profile_end()
    assert twell.twell_get_device_status() == 0
    for fam, n in expect.items():
        assert prof[fam][0] == n, (fam, prof)
    rows = np.array([0, 7, M // 2, M - 1], dtype=np.int64)
    neurons = np.array([0, 5, f // 3, f - 1], dtype=np.int64)
    oracle.set_threads(os.cpu_count() or 1)
    try:
        al = bwd_allowance_sampled(w, lam, rows, neurons)
        dx_ref = oracle.ffn_bwd_dx_rows(w["x"], w["wgT"], w["wuT"], w["wd"], w["dy"], lam, rows)
        og, ou, od = oracle.ffn_bwd_dw_neurons(w["x"], w["wgT"], w["wuT"], w["wd"], w["dy"], lam,
                                               neurons)
    finally:
        oracle.set_threads(1)
    assert_close(to_np(dx)[rows], dx_ref, "dx", out_bf16=True, allowance=al["dx"])
    assert_close(dws[0].cpu().numpy()[neurons], og, "dwgT", allowance=al["dwgT"])
    assert_close(dws[1].cpu().numpy()[neurons], ou, "dwuT", allowance=al["dwuT"])
    assert_close(dws[2].cpu().numpy()[neurons], od, "dwd", allowance=al["dwd"])


def test_neuron_phase_split_when_x_and_dy_exceed_l2():
    """Once x and dY together outgrow 3/4 of L2 the neuron phase runs twice,
    over dY rows for dWd and over x rows for dWu^T and dWg^T; sampled neurons
    against the oracle and the two launches seen by the profiler."""
    from helpers import bwd_allowance_sampled

    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    d, f, lam = 4096, 2048, 2e-5
    M = int(math.ceil(0.75 * l2 / (4 * d) / 128.0)) * 128 + 128
    assert 4.0 * M * d > 0.75 * l2
    w = synthetic.make_inputs(M, d, f, density=0.01, seed=13)
    x, wg, wu, wd, dy = (dev_bf16(w[k]) for k in ("x", "wgT", "wuT", "wd", "dy"))
    shape = twell.make_shape(M, d, f, 128, 32)
    tiles = twell.alloc_tiles(shape)
    twell.twell_pack(x, wg, shape, tiles)
    W = int(twell.tiles_view(tiles, shape)[3].max().item())
    route = twell.alloc_hybrid(shape, W)
    twell.hybrid_route(tiles, shape, route)
    ws = torch.empty(twell.twell_workspace_bytes(shape, W, True), dtype=torch.uint8,
                     device="cuda")
    dx = torch.empty((M, d), dtype=torch.bfloat16, device="cuda")
    dws = [torch.full((f, d), float("nan"), device="cuda") for _ in range(3)]
    twell.twell_profile_begin("*")
    twell.twell_ffn_bwd(x, wg, wu, wd, dy, shape, route, lam, dx, *dws, ws)
    torch.cuda.synchronize()
    prof = twell.twell_profile_end()
    assert twell.twell_get_device_status() == 0
    assert prof["bwd_neurons_dy"][0] == 1 and prof["bwd_neurons_x"][0] == 1, prof
    assert "bwd_neurons" not in prof
    rows = np.array([0, M - 1], dtype=np.int64)
    neurons = np.array([0, 7, f // 2, f - 1], dtype=np.int64)
    oracle.set_threads(os.cpu_count() or 1)
    try:
        al = bwd_allowance_sampled(w, lam, rows, neurons)
        og, ou, od = oracle.ffn_bwd_dw_neurons(w["x"], w["wgT"], w["wuT"], w["wd"], w["dy"], lam,
                                               neurons)
    finally:
        oracle.set_threads(1)
    assert_close(dws[0].cpu().numpy()[neurons], og, "dwgT", allowance=al["dwgT"])
    assert_close(dws[1].cpu().numpy()[neurons], ou, "dwuT", allowance=al["dwuT"])
    assert_close(dws[2].cpu().numpy()[neurons], od, "dwd", allowance=al["dwd"])


def test_multi_pass_twell_split_forward_matches_fused():
    """The TwELL (inference) forward of wide rows with a workspace: the up
    and down gathers each run in L2-sized tile ranges once Wu^T (or Wd) alone
    outgrows 3/4 of L2; a row's h stay in order across the ranges, so y must
    equal the fused single-pass forward bit for bit."""
    d, f = 4096, 16384
    passes = _expected_passes(2.0 * f * d)
    assert passes > 1, "shape no longer exceeds L2; pick a larger one"
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M = 4 * sms + 37  # two rows per team group: no cluster split for the fused forward
    w = synthetic.make_inputs(M, d, f, seed=17, with_dy=False)
    x, wg, wu, wd = (dev_bf16(w[k]) for k in ("x", "wgT", "wuT", "wd"))
    shape = twell.make_shape(M, d, f, 128, 32)
    tiles = twell.alloc_tiles(shape)
    twell.twell_pack(x, wg, shape, tiles)
    y_fused = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    twell.twell_ffn_fwd(x, wg, wu, wd, shape, y_fused, tiles=tiles)
    ws = torch.empty(twell.twell_tiles_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    y_split = torch.full((M, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    twell.twell_profile_begin("*")
    twell.twell_ffn_fwd(x, wg, wu, wd, shape, y_split, tiles=tiles, ws=ws)
    torch.cuda.synchronize()
    prof = twell.twell_profile_end()
    assert twell.twell_get_device_status() == 0
    assert prof["sparse_fwd_up"][0] == passes and prof["sparse_fwd_down"][0] == passes, prof
    assert torch.equal(y_split.view(torch.int16), y_fused.view(torch.int16))


def test_neuron_phase_column_windows_when_x_alone_exceeds_half_of_l2():
    """When x (or dY) alone outgrows half of L2, each neuron pass runs in two
    column windows that gather a column slice of the rows and own their dW
    columns: four launches in all.  Sampled neurons (every column, both
    windows) against the oracle."""
    from helpers import bwd_allowance_sampled

    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    d, f, lam = 4096, 1024, 2e-5
    M = int(math.ceil(0.5 * l2 / (2 * d) / 128.0)) * 128 + 256
    assert 2.0 * M * d > 0.5 * l2
    w = synthetic.make_inputs(M, d, f, density=0.01, seed=14)
    x, wg, wu, wd, dy = (dev_bf16(w[k]) for k in ("x", "wgT", "wuT", "wd", "dy"))
    shape = twell.make_shape(M, d, f, 128, 32)
    tiles = twell.alloc_tiles(shape)
    twell.twell_pack(x, wg, shape, tiles)
    W = int(twell.tiles_view(tiles, shape)[3].max().item())
    route = twell.alloc_hybrid(shape, W, dense_cap=0)
    twell.hybrid_route(tiles, shape, route)
    ws = torch.empty(twell.twell_workspace_bytes(shape, W, True, dense_cap=0), dtype=torch.uint8,
                     device="cuda")
    dx = torch.empty((M, d), dtype=torch.bfloat16, device="cuda")
    dws = [torch.full((f, d), float("nan"), device="cuda") for _ in range(3)]
    twell.twell_profile_begin("*")
    twell.twell_ffn_bwd(x, wg, wu, wd, dy, shape, route, lam, dx, *dws, ws)
    torch.cuda.synchronize()
    prof = twell.twell_profile_end()
    assert twell.twell_get_device_status() == 0
    assert prof["bwd_neurons_dy"][0] == 2 and prof["bwd_neurons_x"][0] == 2, prof
    for t in dws:
        assert torch.isfinite(t).all()  # both windows wrote every column
    rows = np.array([0, M - 1], dtype=np.int64)
    neurons = np.array([0, 3, f // 2, f - 1], dtype=np.int64)
    oracle.set_threads(os.cpu_count() or 1)
    try:
        al = bwd_allowance_sampled(w, lam, rows, neurons)
        og, ou, od = oracle.ffn_bwd_dw_neurons(w["x"], w["wgT"], w["wuT"], w["wd"], w["dy"], lam,
                                               neurons)
    finally:
        oracle.set_threads(1)
    assert_close(dws[0].cpu().numpy()[neurons], og, "dwgT", allowance=al["dwgT"])
    assert_close(dws[1].cpu().numpy()[neurons], ou, "dwuT", allowance=al["dwuT"])
    assert_close(dws[2].cpu().numpy()[neurons], od, "dwd", allowance=al["dwd"])
