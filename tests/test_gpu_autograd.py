"""The PyTorch autograd binding: gradients equal the C ABI's own backward and
the oracle's, and a one-layer training loop with the L1 term on the gate
activations (page 2 "Sakana AI and NVIDIA introduce TwELL with CUDA kernels
...", section "Receta de entrenamiento") drives the gate from ~50 % dense to
sparse while the hybrid router moves rows from the dense fallback to ELL."""
import numpy as np
import pytest
import torch

import oracle
from activation_sparse_gated_tcgen05_gb300 import synthetic, twell
from activation_sparse_gated_tcgen05_gb300.autograd import ell_width_for, sparse_gated_ffn

from helpers import assert_close, dev_bf16, to_np

pytestmark = pytest.mark.gpu
LAM = 2e-5


def test_autograd_matches_abi_and_oracle():
    M, d, f = 300, 256, 1024
    w = synthetic.make_exact_gate_inputs(M, d, f, density=0.02, seed=4, mixed_rows=True)
    x, wg, wu, wd, dy = (dev_bf16(w[k]) for k in ("x", "wgT", "wuT", "wd", "dy"))
    params = [t.clone().requires_grad_() for t in (wg, wu, wd)]
    xr = x.clone().requires_grad_()
    stats = {}
    y = sparse_gated_ffn(xr, *params, l1_coeff=LAM, tile_n=64, tile_cap=16,
                         route_fraction=0.1, stats=stats)
    y.backward(dy)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 0
    assert 0 < stats["routed_rows"] < M
    # the same calls made directly through the binding: identical bytes
    shape = twell.make_shape(M, d, f, 64, 16)
    tiles = twell.alloc_tiles(shape)
    twell.twell_pack(x, wg, shape, tiles)
    W = ell_width_for(twell.tiles_view(tiles, shape)[3], 0.1)
    assert W == stats["ell_width"]
    route = twell.alloc_hybrid(shape, W)
    twell.hybrid_route(tiles, shape, route)
    ws = torch.empty(twell.twell_workspace_bytes(shape, W, True), dtype=torch.uint8,
                     device="cuda")
    y2 = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    twell.twell_ffn_fwd(x, wg, wu, wd, shape, y2, route=route, ws=ws)
    dx2 = torch.empty_like(y2)
    dws2 = [torch.empty(f, d, device="cuda") for _ in range(3)]
    twell.twell_ffn_bwd(x, wg, wu, wd, dy, shape, route, LAM, dx2, *dws2, ws)
    torch.cuda.synchronize()
    assert torch.equal(y.detach().view(torch.int16), y2.view(torch.int16))
    assert torch.equal(xr.grad.view(torch.int16), dx2.view(torch.int16))
    for p, g2 in zip(params, dws2):
        # bf16 parameters receive the fp32 gradient rounded to bf16
        assert torch.equal(p.grad, g2.to(torch.bfloat16))
    ref = oracle.ffn_bwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"], w["dy"], LAM)
    assert_close(to_np(xr.grad), ref["dx"], "dx", out_bf16=True)
    assert_close(dws2[0].cpu().numpy(), ref["dwgT"], "dwgT")


def test_fp32_master_weights_get_fp32_gradients():
    M, d, f = 128, 256, 1024
    w = synthetic.make_inputs(M, d, f, density=0.01, seed=5)
    x, dy = dev_bf16(w["x"]), dev_bf16(w["dy"])
    params = [dev_bf16(w[k]).float().requires_grad_() for k in ("wgT", "wuT", "wd")]
    y = sparse_gated_ffn(x, *params, l1_coeff=LAM, tile_n=64, tile_cap=16, route_fraction=0.0)
    y.backward(dy)
    torch.cuda.synchronize()
    for p in params:
        assert p.grad.dtype == torch.float32 and torch.isfinite(p.grad).all()


def test_one_layer_training_sparsifies_and_unroutes():
    """Student FFN trained against a fixed random teacher with MSE + L1 on the
    gate.  From a dense init (~50 % of gates live, every row overflows its
    tiles and takes the dense fallback) the L1 term drives the gate sparse;
    rows move to the ELL gather as their tiles stop overflowing."""
    torch.manual_seed(0)
    M, d, f, lam = 2048, 256, 1024, 3e-3
    dev = "cuda"

    def batch():
        x = torch.randn(M, d, device=dev)
        x[:, -1] = 1.0
        return x

    tg, tu, td = (torch.randn(f, d, device=dev) * s for s in (d ** -0.5, d ** -0.5, f ** -0.5))
    tg[:, -1] = -2.05 * tg[:, :-1].norm(dim=1)
    torch.manual_seed(1)
    params = [(torch.randn(f, d, device=dev) * s).requires_grad_()
              for s in (d ** -0.5, d ** -0.5, f ** -0.5)]
    opt = torch.optim.Adam(params, lr=1e-3)
    hist = []
    for step in range(200):
        x = batch()
        with torch.no_grad():  # the teacher is plain input data for the student
            yt = (torch.relu(x @ tg.T) * (x @ tu.T)) @ td
        stats = {}
        y = sparse_gated_ffn(x.to(torch.bfloat16), *params, l1_coeff=lam, tile_n=64,
                             tile_cap=16, route_fraction=0.03, stats=stats)
        loss = ((y.float() - yt) ** 2).sum() / M
        opt.zero_grad()
        loss.backward()
        opt.step()
        hist.append((float(loss.item()), stats["density"], stats["routed_rows"]))
    assert twell.twell_get_device_status() == 0
    loss0, dens0, routed0 = hist[0]
    loss1, dens1, routed1 = hist[-1]
    assert np.isfinite([h[0] for h in hist]).all()
    assert dens0 > 0.4 and routed0 == M      # dense start: every row in the fallback
    assert loss1 < 0.1 * loss0
    assert dens1 < 0.05                      # sparse end
    assert routed1 < 0.1 * M                 # most rows back in the ELL gather
