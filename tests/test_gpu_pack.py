"""TwELL packing and hybrid routing on the GPU against the CPU oracle.

Integer and byte outputs (idx, cnt, row_nnz, ELL columns, routed-row list)
must match bit for bit, and so must the bf16 values whenever both sides see
the same pre-activation bytes:
  * twell_pack_dense gets identical fp32 / bf16 input;
  * twell_pack (fused gate GEMM) gets integer-valued inputs whose fp32
    accumulation is exact in any order, so its pre-activation equals the
    oracle's bit for bit.
On real-valued inputs the fused pack is compared with the oracle's fp64
pack: entries agree exactly except where |a| is within the fp32
accumulation error bound of zero (a liveness decision both sides may take
either way), and values agree to one bf16 rounding step."""
import numpy as np
import pytest
import torch

import oracle
from activation_sparse_gated_tcgen05_gb300 import synthetic, twell

from helpers import bf16_bits, dev_bf16

pytestmark = pytest.mark.gpu


def gpu_tiles(shape, tiles):
    val, idx, cnt, nnz = twell.tiles_view(tiles, shape)
    return bf16_bits(val), idx.cpu().numpy(), cnt.cpu().numpy(), nnz.cpu().numpy()


def assert_tiles_equal(got, want, cap):
    gv, gi, gc, gn = got
    wv, wi, wc, wn = want
    np.testing.assert_array_equal(gc, wc)
    np.testing.assert_array_equal(gn, wn)
    stored = np.minimum(wc, cap)
    mask = np.arange(cap)[None, None, :] < stored[:, :, None]  # slots holding data
    np.testing.assert_array_equal(gi[mask], wi[mask])
    np.testing.assert_array_equal(gv[mask], wv[mask])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M,f,tile_n,cap,p", [
    (256, 1024, 64, 16, 0.005), (300, 2048, 128, 32, 0.02), (77, 512, 64, 2, 0.1),
    (129, 1024, 128, 4, 0.05), (1, 256, 128, 128, 0.5)])
def test_pack_dense_bit_exact(dtype, M, f, tile_n, cap, p):
    a = synthetic.make_sparse_preact(M, f, p, seed=M + f)
    if dtype == "bf16":
        a_bits = synthetic.to_bf16_bits(np.nan_to_num(a, nan=1.0))  # bf16 input, keep NaN out
        a_bits[0, 0] = 0x7FC0  # but plant one NaN back
        a_dev = dev_bf16(a_bits)
        a_host = a_bits
    else:
        a_dev = torch.from_numpy(a).cuda()
        a_host = a
    shape = twell.make_shape(M, 64, f, tile_n, cap)
    t = twell.alloc_tiles(shape)
    twell.twell_pack_dense(a_dev, shape, t)
    torch.cuda.synchronize()
    want = oracle.twell_pack(a_host, tile_n, cap)
    assert_tiles_equal(gpu_tiles(shape, t), want, cap)


@pytest.mark.parametrize("M,d,f,tile_n,cap,p", [
    (256, 256, 1024, 64, 16, 0.005),     # tiny config geometry
    (300, 512, 2048, 128, 32, 0.02),     # ragged M, several N tiles
    (1000, 1024, 4096, 128, 4, 0.05),    # overflowing tiles (cnt > C)
    (5, 128, 384, 128, 32, 0.3),         # d_ff not a multiple of 256
    # small batches with K split over a thread-block cluster (the leader sums
    # the other blocks' partials): 2, 8 and 4 splits, the last over two row
    # tiles with a 2-row ragged second tile
    (5, 1024, 1024, 128, 32, 0.05),
    (64, 4096, 2048, 128, 32, 0.02),
    (130, 2048, 1024, 64, 8, 0.1),
])
def test_fused_pack_bit_exact_on_exact_inputs(M, d, f, tile_n, cap, p):
    w = synthetic.make_integer_gate_inputs(M, d, f, density=p, seed=M)
    shape = twell.make_shape(M, d, f, tile_n, cap)
    t = twell.alloc_tiles(shape)
    twell.twell_pack(dev_bf16(w["x"]), dev_bf16(w["wgT"]), shape, t)
    torch.cuda.synchronize()
    assert twell.twell_get_device_status() == 0
    a = oracle.gate_preact(w["x"], w["wgT"])  # exact integers
    want = oracle.twell_pack(a, tile_n, cap)
    assert_tiles_equal(gpu_tiles(shape, t), want, cap)


def test_fused_pack_real_inputs_match_up_to_rounding():
    wl = synthetic.WORKLOADS["tiny_fwd"]
    w = synthetic.make_workload(wl)
    M, d, f, tn, cap = wl.M, wl.d_model, wl.d_ff, wl.tile_n, wl.tile_cap
    shape = twell.make_shape(M, d, f, tn, cap)
    t = twell.alloc_tiles(shape)
    twell.twell_pack(dev_bf16(w["x"]), dev_bf16(w["wgT"]), shape, t)
    torch.cuda.synchronize()
    gv, gi, gc, gn = gpu_tiles(shape, t)
    a = oracle.gate_preact(w["x"], w["wgT"])
    # fp32 accumulation error bound on a: d * 2^-23 * sum_k |x_k w_k|
    xa = np.abs(oracle.f64(w["x"]))
    ga = np.abs(oracle.f64(w["wgT"]))
    bound = d * 2.0 ** -23 * (xa @ ga.T)
    ambiguous = np.abs(a) <= bound
    T = f // tn
    g_live = np.zeros((M, f), bool)
    g_val = np.zeros((M, f))
    for m in range(M):
        for tt in range(T):
            for s in range(min(gc[m, tt], cap)):
                col = tt * tn + int(gi[m, tt, s])
                g_live[m, col] = True
                g_val[m, col] = oracle.f64(gv[m, tt, s:s + 1])[0]
    o_live = oracle.f64(oracle.double_to_bf16(np.maximum(a, 0))) > 0
    assert not (g_live != o_live)[~ambiguous].any()
    both = g_live & o_live
    ref = oracle.f64(oracle.double_to_bf16(np.maximum(a, 0)))
    # one bf16 step = 2^-7 relative at most
    assert (np.abs(g_val[both] - ref[both]) <= 2.0 ** -7 * np.abs(ref[both]) + 1e-30).all()
    assert int(gc.astype(np.int64).sum()) == int(gn.sum())
    assert (gc <= cap).all()


def _upload_tiles(shape, val, idx, cnt, nnz):
    t = twell.alloc_tiles(shape)
    v, i, c, n = twell.tiles_view(t, shape)
    v.copy_(dev_bf16(val))
    i.copy_(torch.from_numpy(idx).cuda())
    c.copy_(torch.from_numpy(cnt).cuda())
    n.copy_(torch.from_numpy(nnz).cuda())
    return t


@pytest.mark.parametrize("W_rule", ["zero", "p90", "inf", "mid"])
def test_route_bit_exact(W_rule):
    M, f, tn, cap = 700, 2048, 128, 8
    a = synthetic.make_sparse_preact(M, f, 0.01, seed=5)
    a[::7] += 1.5  # dense-ish rows, some of them overflow tiles
    val, idx, cnt, nnz = oracle.twell_pack(a, tn, cap)
    W = {"zero": 0, "p90": int(np.sort(nnz)[int(0.9 * M)]), "inf": int(nnz.max()),
         "mid": int(np.median(nnz))}[W_rule]
    shape = twell.make_shape(M, 64, f, tn, cap)
    t = _upload_tiles(shape, val, idx, cnt, nnz)
    h = twell.alloc_hybrid(shape, W)
    twell.hybrid_route(t, shape, h)
    torch.cuda.synchronize()
    ev, ec, en, dr, nd = twell.hybrid_view(h, shape)
    wv, wc, wn, wdr = oracle.hybrid_route(val, idx, cnt, nnz, f, tn, W)
    n = int(nd.item())
    np.testing.assert_array_equal(dr[:n].cpu().numpy(), wdr)
    en = en.cpu().numpy()
    np.testing.assert_array_equal(en, wn)
    if W > 0:
        ev, ec = bf16_bits(ev), ec.cpu().numpy().view(np.uint16)
        mask = np.arange(W)[None, :] < wn[:, None]
        np.testing.assert_array_equal(ec[mask], wc[mask])
        np.testing.assert_array_equal(ev[mask], wv[mask])


def test_route_large_stable_list():
    # more rows than one pass of the list kernel (16384)
    M, f, tn, cap = 40000, 256, 128, 32
    rng = np.random.default_rng(0)
    cnt = rng.integers(0, 6, size=(M, f // tn)).astype(np.uint8)
    nnz = cnt.sum(1).astype(np.int32)
    val = np.full((M, f // tn, cap), 0x3F80, np.uint16)
    idx = np.tile(np.arange(cap, dtype=np.uint8), (M, f // tn, 1))
    shape = twell.make_shape(M, 64, f, tn, cap)
    t = _upload_tiles(shape, val, idx, cnt, nnz)
    W = 5
    h = twell.alloc_hybrid(shape, W)
    twell.hybrid_route(t, shape, h)
    torch.cuda.synchronize()
    _, _, en, dr, nd = twell.hybrid_view(h, shape)
    want = np.nonzero(nnz > W)[0]
    assert int(nd.item()) == want.size
    np.testing.assert_array_equal(dr[: want.size].cpu().numpy(), want)
