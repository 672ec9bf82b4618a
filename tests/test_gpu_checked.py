"""The checked (debug) build, libtwell_checked.so: compiled with
-DTWELL_CHECKED, every index a gather or index kernel reads from memory (ELL
column below d_ff, in-tile column below T_n, ELL length at most W, entry
position below M * W, CSC row below M) is tested before use and a bad one
is reported as TWELL_ERR_INDEX (8) in the device status word instead of
being followed.  Valid inputs: a whole training step matches the oracle
with status 0.  Corrupted indices: the step runs to the end and reports 8.

Each case runs in a child process that loads the checked library
(TWELL_CHECKED=1), since the parent has the normal one loaded."""
import os
import subprocess
import sys

import pytest

from activation_sparse_gated_tcgen05_gb300 import _build

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
import numpy as np
import torch
sys.path.insert(0, {tests!r})
import oracle
from activation_sparse_gated_tcgen05_gb300 import synthetic, twell
from helpers import assert_close, dev_bf16, to_np

assert twell.library_path().endswith("libtwell_checked.so")
LAM = 2e-5
M, d, f, tile_n, cap = {shape}
w = synthetic.make_exact_gate_inputs(M, d, f, density=0.02, seed=5, mixed_rows=True)
x, wg, wu, wd, dy = (dev_bf16(w[k]) for k in ("x", "wgT", "wuT", "wd", "dy"))
shape = twell.make_shape(M, d, f, tile_n, cap)
tiles = twell.alloc_tiles(shape)
twell.twell_pack(x, wg, shape, tiles)
nnz = twell.tiles_view(tiles, shape)[3].cpu().numpy()
W = int(np.sort(nnz)[int(0.8 * (M - 1))])
route = twell.alloc_hybrid(shape, W)
twell.hybrid_route(tiles, shape, route)


def step():
    ws = torch.empty(twell.twell_workspace_bytes(shape, W, True), dtype=torch.uint8, device="cuda")
    y = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    twell.twell_ffn_fwd(x, wg, wu, wd, shape, y, route=route, ws=ws)
    dx = torch.empty_like(y)
    dws = [torch.empty(f, d, device="cuda") for _ in range(3)]
    twell.twell_ffn_bwd(x, wg, wu, wd, dy, shape, route, LAM, dx, *dws, ws)
    torch.cuda.synchronize()
    return y, dx, dws


# uniform-density inputs for the TwELL (inference) forward: no tile overflows
w2 = synthetic.make_exact_gate_inputs(M, d, f, density=0.02, seed=6)
x2, wg2 = dev_bf16(w2["x"]), dev_bf16(w2["wgT"])
t2 = twell.alloc_tiles(shape)
twell.twell_pack(x2, wg2, shape, t2)
mode = {mode!r}
if mode == "valid":
    y, dx, dws = step()
    assert twell.twell_get_device_status() == 0
    assert int(route.n_dense[0].item()) > 0  # routed rows too
    y_ref = oracle.ffn_fwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"])
    ref = oracle.ffn_bwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"], w["dy"], LAM)
    assert_close(to_np(y), y_ref, "y", out_bf16=True)
    assert_close(to_np(dx), ref["dx"], "dx", out_bf16=True)
    assert_close(dws[0].cpu().numpy(), ref["dwgT"], "dwgT")
    assert_close(dws[1].cpu().numpy(), ref["dwuT"], "dwuT")
    assert_close(dws[2].cpu().numpy(), ref["dwd"], "dwd")
    yt = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    tws = twell.twell_tiles_workspace_bytes(shape)
    ws_t = torch.empty(tws, dtype=torch.uint8, device="cuda") if tws else None
    twell.twell_ffn_fwd(x2, wg2, wu, wd, shape, yt, tiles=t2, ws=ws_t)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 0
    yt_ref = oracle.ffn_fwd_dense(w2["x"], w2["wgT"], w["wuT"], w["wd"])
    assert_close(to_np(yt), yt_ref, "y (TwELL)", out_bf16=True)
elif mode == "bad_ell_col":
    _, col, ell_nnz, _, _ = twell.hybrid_view(route, shape)
    m = int(torch.nonzero(ell_nnz > 0)[0].item())
    col[m, 0] = f  # one column past the last neuron
    assert twell.twell_get_device_status() == 0
    step()
    st = twell.twell_get_device_status()
    assert st == 8, st
elif mode == "bad_tile_idx":
    val, idx, cnt, _ = twell.tiles_view(t2, shape)
    assert int(cnt.max().item()) <= cap
    m, t = (int(v) for v in torch.nonzero(cnt > 0)[0])
    idx[m, t, 0] = 255  # past the tile width
    assert twell.twell_get_device_status() == 0
    yt = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    twell.twell_ffn_fwd(x2, wg2, wu, wd, shape, yt, tiles=t2)
    torch.cuda.synchronize()
    st = twell.twell_get_device_status()
    assert st == 8, st
    # routing reads the entries of every row it compacts: with W = d_ff no
    # row is routed for its length, so the corrupted entry is read
    route_all = twell.alloc_hybrid(shape, f)
    twell.hybrid_route(t2, shape, route_all)
    torch.cuda.synchronize()
    st = twell.twell_get_device_status()
    assert st == 8, st
print("child ok")
'''


@pytest.fixture(scope="module")
def checked_lib():
    return _build.build_checked()


def _run(shape, mode):
    env = dict(os.environ, TWELL_CHECKED="1")
    code = CHILD.format(tests=os.path.join(ROOT, "tests"), shape=shape, mode=mode)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "child ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]


# d_model 256 runs the fused gathers, 2048 the split ones
@pytest.mark.parametrize("shape", [(300, 256, 1024, 64, 16), (300, 2048, 1024, 128, 32)])
def test_checked_build_step_matches_oracle(checked_lib, shape):
    _run(shape, "valid")


@pytest.mark.parametrize("shape", [(300, 256, 1024, 64, 16), (300, 2048, 1024, 128, 32)])
@pytest.mark.parametrize("mode", ["bad_ell_col", "bad_tile_idx"])
def test_checked_build_reports_bad_indices(checked_lib, shape, mode):
    _run(shape, mode)
