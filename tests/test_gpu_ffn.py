"""Sparse gated FFN forward / backward and the dense comparator on the GPU,
through the C ABI, against the fp64 CPU oracle on identical seeded inputs.

Tolerance (bf16 in, fp32 accumulate): relative Frobenius error <= 5e-3 and
max |err| <= 2e-2 * rms(ref) on every float output, plus the bf16 storage
rounding (2^-8 |ref|) for outputs stored as bf16; integer outputs exact."""
import numpy as np
import pytest
import torch

import oracle
from activation_sparse_gated_tcgen05_gb300 import synthetic, twell

from helpers import (assert_close, bwd_allowance, dense_intermediate_allowance,
                     dense_silu_intermediate_allowance, dev_bf16, fwd_allowance, to_np)

pytestmark = pytest.mark.gpu
LAM = 2e-5


class Run:
    """Inputs on the device plus the library calls of one step."""

    def __init__(self, M, d, f, tile_n, cap, density=0.005, sigma=None, seed=0, exact=False,
                 mixed=False):
        if exact:
            self.w = synthetic.make_exact_gate_inputs(M, d, f, density=density, seed=seed,
                                                      mixed_rows=mixed)
        else:
            self.w = synthetic.make_inputs(M, d, f, density=density, seed=seed,
                                           lognormal_sigma=sigma)
        self.shape = twell.make_shape(M, d, f, tile_n, cap)
        self.x, self.wg, self.wu, self.wd, self.dy = (
            dev_bf16(self.w[k]) for k in ("x", "wgT", "wuT", "wd", "dy"))
        self.M, self.d, self.f = M, d, f

    def pack(self):
        t = twell.alloc_tiles(self.shape)
        twell.twell_pack(self.x, self.wg, self.shape, t)
        return t

    def route(self, tiles, W):
        h = twell.alloc_hybrid(self.shape, W)
        twell.hybrid_route(tiles, self.shape, h)
        return h

    def fwd(self, tiles=None, route=None, W=0):
        y = torch.empty(self.M, self.d, dtype=torch.bfloat16, device="cuda")
        ws = None
        if route is not None:
            ws = torch.empty(twell.twell_workspace_bytes(self.shape, W, False), dtype=torch.uint8,
                             device="cuda")
        twell.twell_ffn_fwd(self.x, self.wg, self.wu, self.wd, self.shape, y, tiles=tiles,
                            route=route, ws=ws)
        return y

    def bwd(self, route, W):
        ws = torch.empty(twell.twell_workspace_bytes(self.shape, W, True), dtype=torch.uint8,
                         device="cuda")
        dx = torch.empty(self.M, self.d, dtype=torch.bfloat16, device="cuda")
        dws = [torch.full((self.f, self.d), float("nan"), device="cuda") for _ in range(3)]
        twell.twell_ffn_bwd(self.x, self.wg, self.wu, self.wd, self.dy, self.shape, route, LAM,
                            dx, *dws, ws)
        return dx, dws


def _quantile_width(tiles, shape, q):
    nnz = twell.tiles_view(tiles, shape)[3].cpu().numpy()
    return int(np.sort(nnz)[min(len(nnz) - 1, int(q * len(nnz)))])


def test_tiny_inference_forward_from_twell():
    wl = synthetic.WORKLOADS["tiny_fwd"]
    r = Run(wl.M, wl.d_model, wl.d_ff, wl.tile_n, wl.tile_cap)
    t = r.pack()
    y = r.fwd(tiles=t)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 0
    ref = oracle.ffn_fwd_dense(r.w["x"], r.w["wgT"], r.w["wuT"], r.w["wd"])
    assert_close(to_np(y), ref, "y", out_bf16=True, allowance=fwd_allowance(r.w))


def test_tiny_inference_forward_exact_gate():
    wl = synthetic.WORKLOADS["tiny_fwd"]
    r = Run(wl.M, wl.d_model, wl.d_ff, wl.tile_n, wl.tile_cap, exact=True)
    t = r.pack()
    y = r.fwd(tiles=t)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 0
    ref = oracle.ffn_fwd_dense(r.w["x"], r.w["wgT"], r.w["wuT"], r.w["wd"])
    assert_close(to_np(y), ref, "y", out_bf16=True)


def _check_step(r, y, dx, dwg, dwu, dwd, allow, dense_intermediates=False):
    """Compare one fwd + bwd step with the oracle.  allow: add the effect of
    gate rounding decisions (real-valued gate inputs); dense_intermediates:
    add the bf16 rounding of h, u, du, da stored between dense GEMMs."""
    w = r.w
    y_ref = oracle.ffn_fwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"])
    ref = oracle.ffn_bwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"], w["dy"], LAM)
    extra = {}
    if allow:
        extra = dict(bwd_allowance(w, LAM), y=fwd_allowance(w))
    if dense_intermediates:
        for k, v in dense_intermediate_allowance(w, LAM).items():
            extra[k] = extra.get(k, 0.0) + v
    assert_close(to_np(y), y_ref, "y", out_bf16=True, allowance=extra.get("y"))
    assert_close(to_np(dx), ref["dx"], "dx", out_bf16=True, allowance=extra.get("dx"))
    assert_close(to_np(dwg), ref["dwgT"], "dwgT", allowance=extra.get("dwgT"))
    assert_close(to_np(dwu), ref["dwuT"], "dwuT", allowance=extra.get("dwuT"))
    assert_close(to_np(dwd), ref["dwd"], "dwd", allowance=extra.get("dwd"))


@pytest.mark.parametrize("q", [0.0, 0.5, 0.9, 0.97, 1.0])
@pytest.mark.parametrize("tile", [(64, 16), (128, 8)])
def test_hybrid_step_exact_gate(q, tile):
    # mixed per-row densities (~50 %, 2 %, ~0 %): q picks the ELL width, so the
    # split between ELL rows and the dense tensor-core backup varies
    r = Run(300, 256, 1024, tile[0], tile[1], density=0.02, seed=1, exact=True, mixed=True)
    t = r.pack()
    W = _quantile_width(t, r.shape, q) if q > 0 else 0
    h = r.route(t, W)
    y = r.fwd(route=h, W=W)
    dx, (dwg, dwu, dwd) = r.bwd(h, W)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 0
    _check_step(r, y, dx, dwg, dwu, dwd, allow=False)


@pytest.mark.parametrize("q", [0.0, 0.9, 1.0])
def test_hybrid_step_gaussian_inputs(q):
    # lognormal per-row density; gate decisions near a bf16 rounding boundary
    # may go either way, and their effect is bounded from the oracle's data
    r = Run(256, 256, 1024, 64, 16, density=0.01, sigma=1.0, seed=1)
    t = r.pack()
    W = _quantile_width(t, r.shape, q) if q > 0 else 0
    h = r.route(t, W)
    y = r.fwd(route=h, W=W)
    dx, (dwg, dwu, dwd) = r.bwd(h, W)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 0
    _check_step(r, y, dx, dwg, dwu, dwd, allow=True)


def test_backward_is_deterministic():
    r = Run(384, 256, 1024, 64, 16, density=0.02, seed=2, exact=True, mixed=True)
    t = r.pack()
    W = _quantile_width(t, r.shape, 0.8)
    h = r.route(t, W)
    a = r.bwd(h, W)
    b = r.bwd(h, W)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0])
    for u, v in zip(a[1], b[1]):
        assert torch.equal(u, v)


def _bits(t):
    """The tensor's bytes as integers, so equality is bitwise (NaN included)."""
    t = t.contiguous()
    if t.element_size() == 1:
        return t
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32)


@pytest.mark.parametrize("M,d,f", [(700, 512, 2048), (1000, 2048, 1024)])
def test_pair_and_single_gemm_forms_agree(M, d, f):
    """The CTA-pair GEMM form (the default) and the single-CTA form
    (twell_set_pair_gemm(0)) give the same bytes through every epilogue: the
    pack of the gate GEMM, the routed rows' gated / backward-gate / store
    GEMMs, and the dense comparator's forward and backward; each run is also
    checked against the oracle."""
    r = Run(M, d, f, 128, 32, density=0.02, seed=7, exact=True, mixed=True)
    out = {}
    for pair in (True, False):
        prev = twell.twell_set_pair_gemm(pair)
        try:
            t = r.pack()
            W = _quantile_width(t, r.shape, 0.7)
            h = r.route(t, W)
            y = r.fwd(route=h, W=W)
            dx, dws = r.bwd(h, W)
            ws = torch.empty(twell.twell_dense_workspace_bytes(r.shape, True),
                             dtype=torch.uint8, device="cuda")
            yd = torch.empty(r.M, r.d, dtype=torch.bfloat16, device="cuda")
            twell.twell_dense_ffn_fwd(r.x, r.wg, r.wu, r.wd, r.shape, yd, True, ws)
            dxd = torch.empty_like(yd)
            dwsd = [torch.empty(r.f, r.d, device="cuda") for _ in range(3)]
            twell.twell_dense_ffn_bwd(r.x, r.wg, r.wu, r.wd, r.dy, r.shape, LAM, dxd, *dwsd, ws)
            torch.cuda.synchronize()
            assert twell.twell_get_device_status() == 0
        finally:
            twell.twell_set_pair_gemm(prev)
        n_dense = int(h.n_dense[0].item())
        assert n_dense > 0  # the routed rows' GEMMs ran
        out[pair] = [twell.tiles_view(t, r.shape)[2], y, dx, *dws, yd, dxd, *dwsd]
        _check_step(r, y, dx, *dws, allow=False)
    for a, b in zip(out[True], out[False]):
        assert torch.equal(_bits(a), _bits(b))


@pytest.mark.parametrize("M", [300, 1])
def test_dense_comparator_matches_oracle(M):
    r = Run(M, 256, 1024, 64, 16, density=0.05, seed=3, exact=True)
    ws = torch.empty(twell.twell_dense_workspace_bytes(r.shape, True), dtype=torch.uint8,
                     device="cuda")
    y = torch.empty(r.M, r.d, dtype=torch.bfloat16, device="cuda")
    twell.twell_dense_ffn_fwd(r.x, r.wg, r.wu, r.wd, r.shape, y, True, ws)
    dx = torch.empty_like(y)
    dws = [torch.empty(r.f, r.d, device="cuda") for _ in range(3)]
    twell.twell_dense_ffn_bwd(r.x, r.wg, r.wu, r.wd, r.dy, r.shape, LAM, dx, *dws, ws)
    torch.cuda.synchronize()
    _check_step(r, y, dx, *dws, allow=False, dense_intermediates=True)


@pytest.mark.parametrize("M", [300, 1])
def test_dense_silu_comparator_matches_oracle(M):
    """The unmodified SiLU-gated FFN (the comparator the recipe starts from):
    smooth gate, so no gate-decision allowance; h, bf16(a), u, du, da are kept
    in bf16 between the GEMMs like the ReLU comparator's intermediates."""
    w = synthetic.make_inputs(M, 256, 1024, density=0.2, seed=6)
    x, wg, wu, wd, dy = (dev_bf16(w[k]) for k in ("x", "wgT", "wuT", "wd", "dy"))
    shape = twell.make_shape(M, 256, 1024, 64, 16)
    ws = torch.empty(twell.twell_dense_workspace_bytes(shape, True), dtype=torch.uint8,
                     device="cuda")
    y = torch.empty(M, 256, dtype=torch.bfloat16, device="cuda")
    twell.twell_dense_ffn_fwd_act(x, wg, wu, wd, shape, twell.ACT_SILU, y, True, ws)
    dx = torch.empty_like(y)
    dws = [torch.full((1024, 256), float("nan"), device="cuda") for _ in range(3)]
    twell.twell_dense_ffn_bwd_act(x, wg, wu, wd, dy, shape, twell.ACT_SILU, 0.0, dx, *dws, ws)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 0
    y_ref = oracle.ffn_fwd_dense_silu(w["x"], w["wgT"], w["wuT"], w["wd"])
    ref = oracle.ffn_bwd_dense_silu(w["x"], w["wgT"], w["wuT"], w["wd"], w["dy"])
    al = dense_silu_intermediate_allowance(w)
    assert_close(to_np(y), y_ref, "y", out_bf16=True, allowance=al["y"])
    assert_close(to_np(dx), ref["dx"], "dx", out_bf16=True, allowance=al["dx"])
    assert_close(dws[0].cpu().numpy(), ref["dwgT"], "dwgT", allowance=al["dwgT"])
    assert_close(dws[1].cpu().numpy(), ref["dwuT"], "dwuT", allowance=al["dwuT"])
    assert_close(dws[2].cpu().numpy(), ref["dwd"], "dwd", allowance=al["dwd"])


def test_capacity_overflow_is_reported_without_route():
    r = Run(64, 256, 1024, 64, 1, density=0.2, seed=4)
    t = r.pack()
    r.fwd(tiles=t)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 4  # TWELL_ERR_CAPACITY
    assert twell.twell_get_device_status() == 0  # reading clears it


def test_empty_batch_is_a_noop():
    r = Run(1, 256, 1024, 64, 16)
    shape = twell.make_shape(0, 256, 1024, 64, 16)
    t = twell.alloc_tiles(shape)
    twell.twell_pack(r.x, r.wg, shape, t)
    y = torch.empty(1, 256, dtype=torch.bfloat16, device="cuda")
    twell.twell_ffn_fwd(r.x, r.wg, r.wu, r.wd, shape, y, tiles=t)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 0


@pytest.mark.parametrize("M", [1, 16, 64])
def test_small_batch_forward(M):
    r = Run(M, 512, 2048, 128, 32, density=0.02, seed=M, exact=True)
    t = r.pack()
    y = r.fwd(tiles=t)
    torch.cuda.synchronize()
    w = r.w
    assert_close(to_np(y), oracle.ffn_fwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"]), "y",
                 out_bf16=True)


@pytest.mark.parametrize("M,d", [(200, 320), (200, 704), (160, 1088), (96, 3136), (64, 4160)])
def test_d_model_leaving_partial_slabs(M, d):
    """The gathers load without predicates: lanes past d_model read the row's
    first slab against a zero x / dY and their sums are never stored.  These
    d_model values leave partial slabs in the one-warp (d <= 1024), four-warp
    two-slab (d <= 2048), four-warp four-slab (d <= 4096) and eight-warp
    four-slab (d > 4096) team shapes of the forward, row and neuron phases."""
    r = Run(M, d, 1024, 64, 16, density=0.02, seed=8, exact=True)
    y = r.fwd(tiles=r.pack())
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 0
    y_ref = oracle.ffn_fwd_dense(r.w["x"], r.w["wgT"], r.w["wuT"], r.w["wd"])
    assert_close(to_np(y), y_ref, "y (TwELL)", out_bf16=True)
    r = Run(M, d, 1024, 64, 16, density=0.02, seed=9, exact=True, mixed=True)
    t = r.pack()
    W = _quantile_width(t, r.shape, 0.9)
    h = r.route(t, W)
    y = r.fwd(route=h, W=W)
    dx, (dwg, dwu, dwd) = r.bwd(h, W)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 0
    _check_step(r, y, dx, dwg, dwu, dwd, allow=False)


@pytest.mark.parametrize("d", [1024, 2048, 3136, 4160])
def test_many_entries_per_row_and_neuron(d):
    """Rows and neurons with several full 32-entry chunks: the gathers take
    their entries from a 32-lane register in batches, and a batch size that
    does not divide 32 must not wrap around to lane 0 of the same chunk.
    Density 0.25 over d_ff = 256 gives ~64 live entries per row and ~75 live
    rows per neuron, in every team shape of the row and neuron phases."""
    r = Run(300, d, 256, 64, 64, density=0.25, seed=12, exact=True)
    t = r.pack()
    W = _quantile_width(t, r.shape, 1.0)  # no row routed
    h = r.route(t, W)
    y = r.fwd(route=h, W=W)
    dx, (dwg, dwu, dwd) = r.bwd(h, W)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 0
    assert int(twell.hybrid_view(h, r.shape)[4].item()) == 0
    _check_step(r, y, dx, dwg, dwu, dwd, allow=False)


@pytest.mark.parametrize("d,f,tile_n", [(2048, 1024, 128), (3136, 1024, 128), (4096, 2048, 128),
                                        (4160, 1024, 128), (2048, 2560, 64)])
def test_twell_split_forward_matches_fused(d, f, tile_n):
    """TwELL rows wider than 1024 given a workspace run as two gathers (up:
    h per tile slot, down: y).  The dot products and the accumulation order
    are the fused kernel's, so y must equal the fused forward bit for bit,
    and the oracle within tolerance.  M keeps both on one team per row."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M = 4 * sms + 37
    r = Run(M, d, f, tile_n, tile_n // 4, density=0.02, seed=14, exact=True)
    t = r.pack()
    y_fused = r.fwd(tiles=t)
    ws = torch.empty(twell.twell_tiles_workspace_bytes(r.shape), dtype=torch.uint8, device="cuda")
    y_split = torch.full_like(y_fused, float("nan"))
    twell.twell_profile_begin("*")
    twell.twell_ffn_fwd(r.x, r.wg, r.wu, r.wd, r.shape, y_split, tiles=t, ws=ws)
    torch.cuda.synchronize()
    prof = twell.twell_profile_end()
    assert twell.twell_get_device_status() == 0
    assert prof["sparse_fwd_up"][0] == 1 and prof["sparse_fwd_down"][0] == 1, prof
    assert torch.equal(y_split.view(torch.int16), y_fused.view(torch.int16))
    y_ref = oracle.ffn_fwd_dense(r.w["x"], r.w["wgT"], r.w["wuT"], r.w["wd"])
    assert_close(to_np(y_split), y_ref, "y", out_bf16=True)


def test_twell_split_forward_flags_overfull_tiles():
    """The split TwELL forward reads only the C stored entries of a tile and
    flags a tile whose count exceeds C, like the fused forward."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M = 4 * sms + 5
    r = Run(M, 2048, 1024, 64, 2, density=0.2, seed=15, exact=True)
    t = r.pack()
    assert twell.twell_get_device_status() == 0
    y_fused = r.fwd(tiles=t)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 4  # TWELL_ERR_CAPACITY
    ws = torch.empty(twell.twell_tiles_workspace_bytes(r.shape), dtype=torch.uint8, device="cuda")
    y_split = torch.empty_like(y_fused)
    twell.twell_ffn_fwd(r.x, r.wg, r.wu, r.wd, r.shape, y_split, tiles=t, ws=ws)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 4  # TWELL_ERR_CAPACITY
    assert torch.equal(y_split.view(torch.int16), y_fused.view(torch.int16))


@pytest.mark.parametrize("M,d,f,q", [(300, 2048, 1024, 0.9), (300, 2048, 1024, 0.0),
                                     (200, 3136, 1024, 1.0), (256, 4096, 8192, 0.9),
                                     (160, 4160, 1024, 0.9)])
def test_split_and_fused_wide_gathers_agree(M, d, f, q):
    """Rows wider than 1024 run as split gathers by default; with
    twell_set_split_gathers(0) the fused kernels of the pages run instead (h
    never leaves registers).  The forward has the same per-entry arithmetic
    and accumulation order, so y must agree bit for bit (d = 4096, f = 8192
    also runs both in several L2-sized passes, with different pass counts).
    The backward's gradient + dX gather forms u over eight warps per row
    (the fused kernel over its own team) and sums dX per group of 32
    entries, so dX and dW may round differently; each is checked against
    the oracle."""
    r = Run(M, d, f, 128, 32, density=0.02, seed=16, exact=True, mixed=True)
    t = r.pack()
    W = _quantile_width(t, r.shape, q) if q > 0 else 0  # W = 0: every live row routed
    h = r.route(t, W)
    out = {}
    try:
        for split in (True, False):
            twell.twell_set_split_gathers(split)
            twell.twell_profile_begin("*")
            y = r.fwd(route=h, W=W)
            dx, dws = r.bwd(h, W)
            torch.cuda.synchronize()
            prof = twell.twell_profile_end()
            assert twell.twell_get_device_status() == 0
            assert ("sparse_fwd_up" in prof) == split and ("bwd_rows" in prof) != split, prof
            if W == 0:
                assert int(twell.hybrid_view(h, r.shape)[4].item()) > 0
            out[split] = [y.view(torch.int16), dx.view(torch.int16)] + [w.view(torch.int32) for w in dws]
            _check_step(r, y, dx, *dws, allow=False)
    finally:
        twell.twell_set_split_gathers(True)
    assert torch.equal(out[True][0], out[False][0])  # y


@pytest.mark.parametrize("M,d", [(1, 2048), (3, 4096), (17, 3136)])
def test_wide_rows_tiny_batches_training_step(M, d):
    """The split gathers with fewer rows than a block holds (teams and warps
    past the last row leave at once, each team's named barrier its own): a
    full step against the oracle, with and without a routed row."""
    r = Run(M, d, 1024, 128, 32, density=0.05, seed=18, exact=True)
    t = r.pack()
    for q in (1.0, 0.0):
        W = _quantile_width(t, r.shape, q) if q > 0 else 0
        h = r.route(t, W)
        y = r.fwd(route=h, W=W)
        dx, (dwg, dwu, dwd) = r.bwd(h, W)
        torch.cuda.synchronize()
        assert twell.twell_get_device_status() == 0
        _check_step(r, y, dx, dwg, dwu, dwd, allow=False)
