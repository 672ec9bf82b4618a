"""The ELL forward gather split into L2-sized neuron passes.

When the gathered weight rows (Wu^T and Wd, 4 * d_ff * d_model bytes) exceed
about 3/4 of L2, the fused up+down kernel of page 2 "Sakana AI and NVIDIA
introduce TwELL with CUDA kernels ...", section "¿Qué hace distinto a TwELL
frente a ELL clásico?" runs once per neuron chunk and carries y_m between
passes in fp32.  A row's ELL columns ascend, every chunk is a contiguous slice
of it and the per-entry arithmetic and accumulation order are unchanged, so
the result must equal the single-pass TwELL forward bit for bit; sampled
rows are also checked against the oracle."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from activation_sparse_gated_tcgen05_gb300 import synthetic, twell

from helpers import assert_close, dev_bf16, fwd_allowance, to_np

pytestmark = pytest.mark.gpu


def _expected_passes(d, f):
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    gathered = 4.0 * f * d
    return 1 if gathered <= 0.75 * l2 else math.ceil(gathered / (0.5 * l2))


# M large enough that the TwELL forward runs one team per row (batches of
# fewer than two row groups per SM split rows over clusters, which sums in
# another order): d = 4096 has one row per group, d = 2048 two
@pytest.mark.parametrize("rows_per_group,d,f", [(1, 4096, 8192), (2, 2048, 16384)])
def test_multi_pass_forward_matches_single_pass(rows_per_group, d, f):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M = 2 * sms * rows_per_group + 37
    passes = _expected_passes(d, f)
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
    twell.twell_profile_begin("sparse_fwd")
    twell.twell_ffn_fwd(x, wg, wu, wd, shape, y_multi, route=route, ws=ws)
    torch.cuda.synchronize()
    prof = twell.twell_profile_end()
    assert twell.twell_get_device_status() == 0
    assert int(twell.hybrid_view(route, shape)[4].item()) == 0
    assert prof["sparse_fwd"][0] == passes
    # same bytes: entries in the same order, fp32 carried exactly between passes
    assert torch.equal(y_multi.view(torch.int16), y_single.view(torch.int16))
    rows = np.array([0, 1, M // 2, M - 1], dtype=np.int64)
    oracle.set_threads(os.cpu_count() or 1)
    try:
        ref = oracle.ffn_fwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"], rows=rows)
    finally:
        oracle.set_threads(1)
    assert_close(to_np(y_multi)[rows], ref, "y", out_bf16=True, allowance=fwd_allowance(w, rows))


def test_multi_pass_backward_rows():
    """dX over ELL rows in L2-sized passes (Wd, Wu^T, Wg^T rows exceed L2):
    sampled rows of dX and sampled neurons of the weight gradients against
    the oracle, and the pass count seen by the profiler."""
    from helpers import bwd_allowance_sampled

    M, d, f, lam = 256, 4096, 8192, 2e-5
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    gathered = 6.0 * f * d
    passes = 1 if gathered <= 0.5 * l2 else math.ceil(gathered / (0.65 * l2))
    assert passes > 1, "shape no longer exceeds L2; pick a larger one"
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
    twell.twell_profile_begin("bwd_rows")
    twell.twell_ffn_bwd(x, wg, wu, wd, dy, shape, route, lam, dx, *dws, ws)
    torch.cuda.synchronize()
    prof = twell.twell_profile_end()
    assert twell.twell_get_device_status() == 0
    assert prof["bwd_rows"][0] == passes
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
