"""PyTorch autograd binding of the sparse gated FFN.

Forward: gate GEMM with the TwELL pack in its epilogue, hybrid ELL / dense
routing, fused sparse up+down projection.  Backward: the sparse backward with
the L1 term on the gate activations (page 2 "Sakana AI and NVIDIA introduce
TwELL with CUDA kernels ...", sections "¿Qué hace distinto a TwELL frente a
ELL clásico?" and "Receta de entrenamiento").  This module only marshals
arguments to the C ABI (twell.py); every step runs in the library's kernels.

Weights are neuron-major [d_ff][d_model] (WgT, WuT, Wd).  They may be fp32
master parameters: the bf16 copies the kernels read are made here, and the
library's fp32 weight gradients are returned unrounded.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import twell


def ell_width_for(row_nnz: torch.Tensor, route_fraction: float) -> int:
    """ELL width W that routes about `route_fraction` of the rows to the dense
    fallback: the row count at sorted index floor((1 - route_fraction) * M)
    (the widest row when route_fraction = 0).  Reads the counts on the host."""
    M = row_nnz.numel()
    if M == 0:
        return 0
    s = torch.sort(row_nnz.to(torch.int64)).values
    if route_fraction <= 0:
        return int(s[-1].item())
    return int(s[min(M - 1, int((1.0 - route_fraction) * M))].item())


class SparseGatedFFNFunction(torch.autograd.Function):
    """y = (ReLU(x Wg) * (x Wu)) Wd with the gate packed into TwELL and
    consumed sparsely; backward adds l1_coeff to dL/da at every live entry."""

    @staticmethod
    def forward(ctx, x, wgT, wuT, wd, l1_coeff: float, tile_n: int, tile_cap: int,
                route_fraction: float, stats: Optional[dict]):
        if x.dim() != 2:
            raise ValueError("x must be [tokens][d_model]")
        M, d = x.shape
        f = wgT.shape[0]
        xb = x.to(torch.bfloat16).contiguous()
        wg, wu, wdb = (w.detach().to(torch.bfloat16).contiguous() for w in (wgT, wuT, wd))
        shape = twell.make_shape(M, d, f, tile_n, tile_cap)
        tiles = twell.alloc_tiles(shape, x.device)
        twell.twell_pack(xb, wg, shape, tiles)
        row_nnz = twell.tiles_view(tiles, shape)[3]
        W = ell_width_for(row_nnz, route_fraction)
        route = twell.alloc_hybrid(shape, W, x.device)
        twell.hybrid_route(tiles, shape, route)
        # the routed-row count is on the device: read it and size the
        # workspace's dense-backup buffers for exactly those rows
        n_dense = int(route.n_dense[0].item())
        route.dense_cap = n_dense
        ws = torch.empty(twell.twell_workspace_bytes(shape, W, True, dense_cap=n_dense),
                         dtype=torch.uint8, device=x.device)
        y = torch.empty(M, d, dtype=torch.bfloat16, device=x.device)
        twell.twell_ffn_fwd(xb, wg, wu, wdb, shape, y, route=route, ws=ws)
        if stats is not None:
            stats["density"] = float(row_nnz.to(torch.float64).sum().item()) / max(1, M * f)
            stats["ell_width"] = W
            stats["routed_rows"] = n_dense
            stats["workspace_bytes"] = ws.numel()
        ctx.save_for_backward(xb, wg, wu, wdb)
        ctx.shape, ctx.route, ctx.ws, ctx.l1 = shape, route, ws, float(l1_coeff)
        ctx.in_dtypes = (x.dtype, wgT.dtype, wuT.dtype, wd.dtype)
        return y

    @staticmethod
    def backward(ctx, dy):
        xb, wg, wu, wdb = ctx.saved_tensors
        shape = ctx.shape
        dyb = dy.to(torch.bfloat16).contiguous()
        dx = torch.empty_like(xb)
        f, d = shape.d_ff, shape.d_model
        dws = [torch.empty(f, d, dtype=torch.float32, device=xb.device) for _ in range(3)]
        twell.twell_ffn_bwd(xb, wg, wu, wdb, dyb, shape, ctx.route, ctx.l1, dx, *dws, ctx.ws)
        xt, gt, ut, dt = ctx.in_dtypes
        grads = [g if g.dtype == t else g.to(t) for g, t in zip(dws, (gt, ut, dt))]
        return (dx if dx.dtype == xt else dx.to(xt), *grads, None, None, None, None, None)


def sparse_gated_ffn(x, wgT, wuT, wd, l1_coeff: float = 2e-5, tile_n: int = 128,
                     tile_cap: int = 32, route_fraction: float = 0.03,
                     stats: Optional[dict] = None):
    """Functional form; `stats`, if given, receives the gate density, the ELL
    width and the number of routed rows of this call (host reads)."""
    return SparseGatedFFNFunction.apply(x, wgT, wuT, wd, l1_coeff, tile_n, tile_cap,
                                        route_fraction, stats)
