"""The gate GEMM + TwELL pack of small batches (M <= 64 tokens), which runs
with the operands swapped: neurons on the MMA's M dimension, tokens on its N
dimension (padded to 16, 32 or 64), K split over a thread-block cluster
whose blocks sum their partials in rank order, and the pack done across
TMEM lanes (one warp ballot per token and warp, counts combined over the
four epilogue warps).

On integer-valued gate inputs (fp32 accumulation exact in any order) the
packed values, in-tile columns, counts and row totals must equal the
oracle's packer bit for bit -- including tiles that overflow their capacity,
T_n = 64 (two TwELL tiles per 128-neuron MMA tile), every token padding
(16 / 32 / 64) and cluster sizes 1 to 8.  The forward on real-valued inputs
at the 8B-class shape is checked against the oracle in
test_gpu_full_size.py."""
import numpy as np
import pytest
import torch

import oracle
from activation_sparse_gated_tcgen05_gb300 import synthetic, twell

from helpers import assert_close, dev_bf16, fwd_allowance, to_np
from test_gpu_pack import assert_tiles_equal, gpu_tiles

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,d,f,tile_n,cap,p,mixed", [
    (1, 4096, 14336, 128, 32, 0.005, False),   # one token, 8B-class shape, 4-way K split
    (3, 4096, 2048, 128, 32, 0.02, False),     # 8-way K split (16 neuron tiles)
    (16, 1024, 4096, 64, 16, 0.02, False),     # T_n = 64: two TwELL tiles per MMA tile
    (17, 512, 1024, 128, 32, 0.05, True),      # 32-token padding, mixed-density rows
    (33, 256, 1024, 64, 4, 0.05, False),       # 64-token padding, overflowing tiles
    (48, 128, 384, 128, 32, 0.3, True),        # one K split, d_ff = 3 tiles
    (64, 4096, 14336, 128, 32, 0.005, True),   # the largest small batch, 8B-class shape
    (64, 2048, 8192, 64, 8, 0.02, False),
])
def test_small_batch_pack_bit_exact(M, d, f, tile_n, cap, p, mixed):
    w = synthetic.make_integer_gate_inputs(M, d, f, density=p, seed=M + d, mixed_rows=mixed)
    shape = twell.make_shape(M, d, f, tile_n, cap)
    t = twell.alloc_tiles(shape)
    # stale bytes in every buffer: the pack must write all it is responsible for
    for buf in (t.val.view(torch.int16), t.idx, t.cnt, t.row_nnz):
        buf.fill_(-1 if buf.dtype != torch.uint8 else 255)
    twell.twell_pack(dev_bf16(w["x"]), dev_bf16(w["wgT"]), shape, t)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 0
    a = oracle.gate_preact(w["x"], w["wgT"])  # exact integers
    want = oracle.twell_pack(a, tile_n, cap)
    assert_tiles_equal(gpu_tiles(shape, t), want, cap)


def test_small_batch_pack_twice_is_stable():
    # two packs in a row into the same buffers give the same bytes
    M, d, f = 16, 2048, 4096
    w = synthetic.make_integer_gate_inputs(M, d, f, density=0.01, seed=9)
    shape = twell.make_shape(M, d, f, 128, 32)
    t = twell.alloc_tiles(shape)
    x, wg = dev_bf16(w["x"]), dev_bf16(w["wgT"])
    twell.twell_pack(x, wg, shape, t)
    first = [b.clone() for b in (t.val, t.idx, t.cnt, t.row_nnz)]
    twell.twell_pack(x, wg, shape, t)
    torch.cuda.synchronize()
    assert torch.equal(first[2], t.cnt) and torch.equal(first[3], t.row_nnz)
    want = oracle.twell_pack(oracle.gate_preact(w["x"], w["wgT"]), 128, 32)
    assert_tiles_equal(gpu_tiles(shape, t), want, 32)


@pytest.mark.parametrize("M", [1, 3, 16, 64])
@pytest.mark.parametrize("with_ws", [False, True])
def test_small_batch_forward_matches_oracle(M, with_ws):
    # real-valued inputs at a mid-size shape: the TwELL forward of the packed
    # small batch against the oracle (gate decisions within the fp32 band),
    # with and without the forward's optional workspace (a small batch runs
    # a cluster of blocks per row either way)
    d, f = 2048, 8192
    w = synthetic.make_inputs(M, d, f, density=0.005, seed=21, with_dy=False)
    x, wg, wu, wd = (dev_bf16(w[k]) for k in ("x", "wgT", "wuT", "wd"))
    shape = twell.make_shape(M, d, f, 128, 32)
    t = twell.alloc_tiles(shape)
    twell.twell_pack(x, wg, shape, t)
    y = torch.full((M, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = (torch.empty(twell.twell_tiles_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
          if with_ws else None)
    twell.twell_ffn_fwd(x, wg, wu, wd, shape, y, tiles=t, ws=ws)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 0
    ref = oracle.ffn_fwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"])
    assert_close(to_np(y), ref, "y", out_bf16=True, allowance=fwd_allowance(w))


@pytest.mark.parametrize("M,d,f,tile_n,cap", [(5, 3136, 1024, 128, 32), (40, 2048, 2560, 64, 16)])
def test_small_batch_forward_exact_gate(M, d, f, tile_n, cap):
    # integer gate inputs (both sides take the same gate decisions): the
    # small-batch forward against the oracle with the plain tolerance, on a
    # d_model that leaves a partial 256-column slab and on T_n = 64
    w = synthetic.make_exact_gate_inputs(M, d, f, density=0.03, seed=M)
    x, wg, wu, wd = (dev_bf16(w[k]) for k in ("x", "wgT", "wuT", "wd"))
    shape = twell.make_shape(M, d, f, tile_n, cap)
    t = twell.alloc_tiles(shape)
    twell.twell_pack(x, wg, shape, t)
    assert int(twell.tiles_view(t, shape)[2].max().item()) <= cap
    y = torch.full((M, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(twell.twell_tiles_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    twell.twell_ffn_fwd(x, wg, wu, wd, shape, y, tiles=t, ws=ws)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 0
    ref = oracle.ffn_fwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"])
    assert_close(to_np(y), ref, "y", out_bf16=True)


def test_small_batch_forward_flags_overfull_tiles():
    # a tile with more live columns than its capacity: the stored entries
    # are used and TWELL_ERR_CAPACITY is recorded, as in every TwELL forward
    M, d, f = 8, 2048, 1024
    w = synthetic.make_exact_gate_inputs(M, d, f, density=0.3, seed=2)
    x, wg, wu, wd = (dev_bf16(w[k]) for k in ("x", "wgT", "wuT", "wd"))
    shape = twell.make_shape(M, d, f, 128, 4)
    t = twell.alloc_tiles(shape)
    twell.twell_pack(x, wg, shape, t)
    assert int(twell.tiles_view(t, shape)[2].max().item()) > 4
    y = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(twell.twell_tiles_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    twell.twell_ffn_fwd(x, wg, wu, wd, shape, y, tiles=t, ws=ws)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 4
    assert torch.isfinite(y.float()).all()
