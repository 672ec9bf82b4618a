"""Pins for the CPU oracle: each test ties the oracle to something other than
itself -- a hand-worked example, an independent library (torch fp64 autograd,
torch's bf16 conversion), finite differences, brute force or a closed form.

All of these run on the CPU (no ``gpu`` marker).
"""
import fractions
import os

import numpy as np
import pytest
import torch

import oracle
from activation_sparse_gated_tcgen05_gb300 import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------- bf16
def _bf16_nearest_even(v: float) -> int:
    """Brute-force bf16 rounding of a double with exact rational arithmetic."""
    if v == 0.0:
        return 0x8000 if np.signbit(v) else 0
    sign = 0x8000 if v < 0 else 0
    a = fractions.Fraction(abs(v))
    # candidate finite positive bf16 values bracketing a
    best = None
    for bits in _bracket(abs(v)):
        fv = fractions.Fraction(float(synthetic.bf16_bits_to_f32(np.array([bits], np.uint16))[0]))
        key = (abs(fv - a), bits & 1)  # nearer first, then even mantissa
        if best is None or key < best[0]:
            best = (key, bits)
    return sign | best[1]


def _bracket(a: float):
    f32 = np.float32(a)
    hi = int(np.array([f32], np.float32).view(np.uint32)[0]) >> 16
    return [b for b in (hi - 1, hi, hi + 1, hi + 2) if 0 <= b < 0x7F80]


def test_bf16_rounding_matches_brute_force_and_torch():
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.standard_normal(300) * 10.0 ** rng.integers(-40, 38, 300),
        rng.standard_normal(100) * 1e-39,            # bf16 subnormal range
        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -40]),  # ties
    ])
    got = oracle.double_to_bf16(v)
    want = np.array([_bf16_nearest_even(float(t)) for t in v], np.uint16)
    np.testing.assert_array_equal(got, want)
    # float32 inputs: the library routine (torch) rounds fp32 -> bf16 to nearest even
    v32 = rng.standard_normal(5000).astype(np.float32) * np.float32(3.0)
    t = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.double_to_bf16(v32.astype(np.float64)), t)


# --------------------------------------------------------------- golden files
def _read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            rows.setdefault(key, []).append(rest)
    return rows


def test_pack_and_route_worked_example():
    g = _read_golden("twell_pack_worked_example.txt")
    tile_n = int(g["tile_n"][0][0])
    cap = int(g["cap"][0][0])
    a = np.array([[float(v) for v in r] for r in g["a"]])
    val, idx, cnt, nnz = oracle.twell_pack(a, tile_n, cap)
    for r in g["tile"]:
        m, t, c = int(r[0]), int(r[1]), int(r[3])
        assert cnt[m, t] == c
        pairs = [p.split(":") for p in r[4:]]
        for s, (i, v) in enumerate(pairs):
            assert idx[m, t, s] == int(i)
            assert oracle.f64(val[m, t, s:s + 1])[0] == float(v)
    np.testing.assert_array_equal(nnz, [int(v) for v in g["row_nnz"][0]])
    for r in g["route"]:
        W = int(r[1])
        k = r.index("dense_rows")
        end = r.index("ell") if "ell" in r else len(r)
        want_dense = [int(v) for v in r[k + 1:end]]
        ev, ec, en, dr = oracle.hybrid_route(val, idx, cnt, nnz, a.shape[1], tile_n, W)
        assert list(dr) == want_dense
        if "ell" in r:
            e = r.index("ell")
            m = int(r[e + 1])
            pairs = [p.split(":") for p in r[e + 2:]]
            assert en[m] == len(pairs)
            for s, (col, v) in enumerate(pairs):
                assert ec[m, s] == int(col)
                assert oracle.f64(ev[m, s:s + 1])[0] == float(v)
        for m in want_dense:
            assert en[m] == 0


def test_ffn_worked_example():
    g = _read_golden("ffn_worked_example.txt")
    arr = lambda k: np.array([[float(v) for v in r] for r in g[k]])
    x, wgT, wuT, wd, dy = arr("x"), arr("wgT"), arr("wuT"), arr("wd"), arr("dy")
    lam = float(g["lambda"][0][0])
    y = oracle.ffn_fwd_dense(x, wgT, wuT, wd)
    np.testing.assert_array_equal(y, arr("y"))
    b = oracle.ffn_bwd_dense(x, wgT, wuT, wd, dy, lam)
    np.testing.assert_array_equal(b["dx"], arr("dx"))
    np.testing.assert_array_equal(b["dwd"], arr("dwd"))
    np.testing.assert_array_equal(b["dwuT"], arr("dwuT"))
    np.testing.assert_array_equal(b["dwgT"], arr("dwgT"))
    assert b["l1"] == float(g["l1"][0][0])
    # the per-row / per-neuron sampled routines give the same numbers
    np.testing.assert_array_equal(oracle.ffn_bwd_dx_rows(x, wgT, wuT, wd, dy, lam, [0]), arr("dx"))
    og, ou, od = oracle.ffn_bwd_dw_neurons(x, wgT, wuT, wd, dy, lam, [0, 1])
    np.testing.assert_array_equal(og, arr("dwgT"))
    np.testing.assert_array_equal(ou, arr("dwuT"))
    np.testing.assert_array_equal(od, arr("dwd"))


# ------------------------------------------------- independent library: torch
def _torch_ffn(x, wgT, wuT, wd, dy, lam):
    X = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    Wg = torch.tensor(wgT.T.copy(), dtype=torch.float64, requires_grad=True)
    Wu = torch.tensor(wuT.T.copy(), dtype=torch.float64, requires_grad=True)
    Wd = torch.tensor(wd, dtype=torch.float64, requires_grad=True)
    a = X @ Wg
    g = torch.relu(a)
    y = (g * (X @ Wu)) @ Wd
    loss = (y * torch.tensor(dy, dtype=torch.float64)).sum() + lam * g.sum()
    loss.backward()
    return (y.detach().numpy(), X.grad.numpy(), Wg.grad.numpy().T, Wu.grad.numpy().T,
            Wd.grad.numpy(), (lam * g.sum()).item(), a.detach().numpy())


@pytest.mark.parametrize("density", [0.1, 0.5, 1.0])
def test_dense_fwd_bwd_match_torch_autograd(density):
    rng = np.random.default_rng(7)
    M, d, f, lam = 12, 16, 24, 2e-2
    x = rng.standard_normal((M, d))
    wgT = rng.standard_normal((f, d)) / 4
    shift = {0.1: -1.0, 0.5: 0.0, 1.0: 50.0}[density]
    x[:, -1] = 1.0
    wgT[:, -1] = shift
    wuT = rng.standard_normal((f, d)) / 4
    wd = rng.standard_normal((f, d)) / 5
    dy = rng.standard_normal((M, d))
    y_t, dx_t, dwg_t, dwu_t, dwd_t, l1_t, a = _torch_ffn(x, wgT, wuT, wd, dy, lam)
    assert np.abs(a).min() > 1e-9  # no kink ties
    y = oracle.ffn_fwd_dense(x, wgT, wuT, wd, round_g=False)
    np.testing.assert_allclose(y, y_t, rtol=1e-12, atol=1e-12)
    b = oracle.ffn_bwd_dense(x, wgT, wuT, wd, dy, lam, round_g=False)
    for got, want in ((b["dx"], dx_t), (b["dwgT"], dwg_t), (b["dwuT"], dwu_t), (b["dwd"], dwd_t)):
        np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-11)
    assert abs(b["l1"] - l1_t) <= 1e-12 * max(1.0, abs(l1_t))
    if density == 1.0:
        assert (a > 0).all()


def test_gate_preact_matches_fp64_matmul_and_a_hand_case():
    # the gate pre-activation a = x Wg (Wg stored neuron-major as Wg^T) on
    # its own: a 2 x 3 case worked by hand, then random inputs against
    # torch's fp64 matmul (a library routine the C++ oracle does not use)
    x = np.array([[1.0, 2.0, -1.0], [0.5, 0.0, 4.0]])
    wgT = np.array([[1.0, 0.0, 0.0], [2.0, -1.0, 3.0], [0.0, 0.25, 0.5], [-1.0, -1.0, -1.0]])
    want = np.array([[1.0, -3.0, 0.0, -2.0], [0.5, 13.0, 2.0, -4.5]])
    np.testing.assert_array_equal(oracle.gate_preact(x, wgT), want)
    rng = np.random.default_rng(21)
    x = rng.standard_normal((37, 48))
    wgT = rng.standard_normal((70, 48))
    ref = (torch.from_numpy(x) @ torch.from_numpy(wgT).t()).numpy()
    np.testing.assert_allclose(oracle.gate_preact(x, wgT), ref, rtol=1e-13, atol=1e-13)


def test_all_dead_gate_gives_exact_zeros():
    rng = np.random.default_rng(3)
    M, d, f = 8, 16, 32
    x = rng.standard_normal((M, d))
    x[:, -1] = 1.0
    wgT = rng.standard_normal((f, d)) / 8
    wgT[:, -1] = -100.0
    wuT = rng.standard_normal((f, d))
    wd = rng.standard_normal((f, d))
    dy = rng.standard_normal((M, d))
    assert not oracle.ffn_fwd_dense(x, wgT, wuT, wd).any()
    b = oracle.ffn_bwd_dense(x, wgT, wuT, wd, dy, 2e-5)
    for k in ("dx", "dwgT", "dwuT", "dwd"):
        assert not b[k].any()
    assert b["l1"] == 0.0


# ----------------------------------------------------------- finite differences
def _loss(x, wgT, wuT, wd, dy, lam):
    y = oracle.ffn_fwd_dense(x, wgT, wuT, wd, round_g=False)
    a = oracle.gate_preact(x, wgT)
    return float((y * dy).sum() + lam * np.maximum(a, 0.0).sum())


def test_backward_matches_finite_differences():
    rng = np.random.default_rng(11)
    M, d, f, lam = 4, 8, 16, 2e-2
    for _ in range(100):  # redraw until every pre-activation is away from the kink
        x = rng.standard_normal((M, d))
        wgT = rng.standard_normal((f, d)) / 2
        if np.abs(oracle.gate_preact(x, wgT)).min() > 1e-3:
            break
    wuT = rng.standard_normal((f, d)) / 2
    wd = rng.standard_normal((f, d)) / 2
    dy = rng.standard_normal((M, d))
    b = oracle.ffn_bwd_dense(x, wgT, wuT, wd, dy, lam, round_g=False)
    h = 1e-6
    names = {"dx": x, "dwgT": wgT, "dwuT": wuT, "dwd": wd}
    for gname, arr in names.items():
        for flat in range(arr.size):
            i = np.unravel_index(flat, arr.shape)
            old = arr[i]
            arr[i] = old + h
            lp = _loss(x, wgT, wuT, wd, dy, lam)
            arr[i] = old - h
            lm = _loss(x, wgT, wuT, wd, dy, lam)
            arr[i] = old
            fd = (lp - lm) / (2 * h)
            an = b[gname][i]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (gname, i, fd, an)


def test_l1_only_closed_form():
    """dY = 0 leaves only the L1 subgradient: dWg^T = lambda * 1[a>0]^T x,
    dx = lambda * 1[a>0] Wg^T, dWu = dWd = 0."""
    rng = np.random.default_rng(5)
    M, d, f, lam = 10, 12, 20, 2e-5
    x = rng.standard_normal((M, d))
    wgT = rng.standard_normal((f, d))
    wuT = rng.standard_normal((f, d))
    wd = rng.standard_normal((f, d))
    b = oracle.ffn_bwd_dense(x, wgT, wuT, wd, np.zeros((M, d)), lam, round_g=False)
    live = (x @ wgT.T > 0).astype(np.float64)
    np.testing.assert_allclose(b["dwgT"], lam * live.T @ x, rtol=1e-12, atol=1e-18)
    np.testing.assert_allclose(b["dx"], lam * live @ wgT, rtol=1e-12, atol=1e-18)
    assert not b["dwuT"].any() and not b["dwd"].any()


# --------------------------------------------------------------- pack (brute)
@pytest.mark.parametrize("cap", [0, 4, 16])
def test_pack_all_sign_patterns_of_a_16_wide_tile(cap):
    pats = np.arange(1 << 16, dtype=np.int64)
    bits = ((pats[:, None] >> np.arange(16)) & 1).astype(bool)
    mag = np.arange(1, 17, dtype=np.float64) * 0.5
    a = np.where(bits, mag, -mag)
    val, idx, cnt, nnz = oracle.twell_pack(a, 16, cap)
    pop = bits.sum(1)
    np.testing.assert_array_equal(cnt[:, 0], pop)
    np.testing.assert_array_equal(nnz, pop)
    # expected slots: the positions of the set bits, ascending, first `cap`
    order = np.where(bits, np.arange(16), 99)
    order.sort(axis=1)
    for s in range(cap):
        has = pop > s
        np.testing.assert_array_equal(idx[has, 0, s], order[has, s])
        np.testing.assert_array_equal(oracle.f64(val[has, 0, s]), mag[order[has, s]])
        assert not idx[~has, 0, s].any() and not val[~has, 0, s].any()


def test_pack_unpack_roundtrip_and_count():
    a = synthetic.make_sparse_preact(64, 512, 0.05, seed=4).astype(np.float64)
    for tile_n in (64, 128):
        val, idx, cnt, nnz = oracle.twell_pack(a, tile_n, tile_n)  # C = T_n: never overflows
        g = oracle.twell_unpack(val, idx, cnt, 512, tile_n)
        # bf16(ReLU(a)) through torch's converter (fp32 input is exact for these values)
        ref = torch.from_numpy(np.maximum(np.nan_to_num(a, nan=0.0, posinf=np.inf, neginf=-np.inf), 0.0).astype(np.float32))
        ref = ref.to(torch.bfloat16).double().numpy()
        np.testing.assert_array_equal(g, ref)
        assert int(cnt.astype(np.int64).sum()) == int((ref > 0).sum())
        np.testing.assert_array_equal(nnz, (ref > 0).sum(1))


# -------------------------------------------------------------------- route
def test_route_extremes_and_equivalence():
    w = synthetic.make_inputs(48, 64, 256, density=0.05, seed=9)
    a = oracle.gate_preact(w["x"], w["wgT"])
    tile_n, cap = 64, 4
    val, idx, cnt, nnz = oracle.twell_pack(a, tile_n, cap)
    overflow = (cnt > cap).any(1)
    # W = infinity: only overflowing rows are routed
    ev, ec, en, dr = oracle.hybrid_route(val, idx, cnt, nnz, 256, tile_n, int(nnz.max()))
    np.testing.assert_array_equal(dr, np.nonzero(overflow)[0])
    # W = 0: every row with a live entry is routed
    _, _, en0, dr0 = oracle.hybrid_route(val, idx, cnt, nnz, 256, tile_n, 0)
    np.testing.assert_array_equal(dr0, np.nonzero(nnz > 0)[0])
    assert not en0.any()
    # ELL rows hold exactly the unpacked live entries, ascending global column
    g = np.maximum(a, 0)
    for m in range(48):
        if m in set(dr.tolist()):
            assert en[m] == 0
            continue
        cols = ec[m, :en[m]].astype(np.int64)
        np.testing.assert_array_equal(cols, np.nonzero(oracle.f64(oracle.double_to_bf16(g[m])) > 0)[0])
    # the forward result does not depend on W
    y_ref = oracle.ffn_fwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"])
    for W in (0, 3, 6, int(nnz.max())):
        ev, ec, en, dr = oracle.hybrid_route(val, idx, cnt, nnz, 256, tile_n, W)
        y = oracle.ffn_fwd_ell(w["x"], w["wuT"], w["wd"], ev, ec, en)
        if dr.size:
            y[dr] = oracle.ffn_fwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"], rows=dr)
        np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------ sparse == dense restatements
def test_sparse_restatements_equal_dense():
    w = synthetic.make_inputs(40, 64, 256, density=0.03, seed=2)
    lam = 2e-5
    a = oracle.gate_preact(w["x"], w["wgT"])
    val, idx, cnt, nnz = oracle.twell_pack(a, 64, 64)
    y_d = oracle.ffn_fwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"])
    y_t = oracle.ffn_fwd_twell(w["x"], w["wuT"], w["wd"], val, idx, cnt, 64)
    np.testing.assert_allclose(y_t, y_d, rtol=1e-12, atol=1e-13)
    b_d = oracle.ffn_bwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"], w["dy"], lam)
    for W in (0, 2, int(nnz.max())):
        val2, idx2, cnt2, nnz2 = oracle.twell_pack(a, 64, 2)
        ev, ec, en, dr = oracle.hybrid_route(val2, idx2, cnt2, nnz2, 256, 64, W)
        b_h = oracle.ffn_bwd_hybrid(w["x"], w["wgT"], w["wuT"], w["wd"], w["dy"], ev, ec, en, dr,
                                    lam)
        for k in ("dx", "dwgT", "dwuT", "dwd"):
            np.testing.assert_allclose(b_h[k], b_d[k], rtol=1e-11, atol=1e-13)
    rows = np.array([0, 7, 39])
    np.testing.assert_allclose(
        oracle.ffn_bwd_dx_rows(w["x"], w["wgT"], w["wuT"], w["wd"], w["dy"], lam, rows),
        b_d["dx"][rows], rtol=1e-12, atol=1e-14)
    neu = np.array([1, 100, 255])
    og, ou, od = oracle.ffn_bwd_dw_neurons(w["x"], w["wgT"], w["wuT"], w["wd"], w["dy"], lam, neu)
    np.testing.assert_allclose(og, b_d["dwgT"][neu], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(ou, b_d["dwuT"][neu], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(od, b_d["dwd"][neu], rtol=1e-12, atol=1e-14)


def test_threads_do_not_change_results():
    w = synthetic.make_inputs(33, 64, 128, density=0.1, seed=6)
    rows = np.arange(33)
    oracle.set_threads(1)
    y1 = oracle.ffn_fwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"], rows=rows)
    oracle.set_threads(5)
    y5 = oracle.ffn_fwd_dense(w["x"], w["wgT"], w["wuT"], w["wd"], rows=rows)
    oracle.set_threads(1)
    np.testing.assert_array_equal(y1, y5)


# ------------------------------------------- SiLU-gated comparator (dense only)
def test_silu_fwd_bwd_match_torch_autograd():
    """The SiLU-gated FFN against torch's own silu and autograd in fp64."""
    rng = np.random.default_rng(21)
    M, d, f = 6, 16, 24
    x = rng.standard_normal((M, d))
    wgT, wuT, wd = (rng.standard_normal((f, d)) / 3 for _ in range(3))
    dy = rng.standard_normal((M, d))
    X = torch.tensor(x, requires_grad=True)
    Wg = torch.tensor(wgT.T.copy(), requires_grad=True)
    Wu = torch.tensor(wuT.T.copy(), requires_grad=True)
    Wd = torch.tensor(wd, requires_grad=True)
    y_t = (torch.nn.functional.silu(X @ Wg) * (X @ Wu)) @ Wd
    (y_t * torch.tensor(dy)).sum().backward()
    y = oracle.ffn_fwd_dense_silu(x, wgT, wuT, wd)
    b = oracle.ffn_bwd_dense_silu(x, wgT, wuT, wd, dy)
    np.testing.assert_allclose(y, y_t.detach().numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b["dx"], X.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b["dwgT"], Wg.grad.numpy().T, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b["dwuT"], Wu.grad.numpy().T, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b["dwd"], Wd.grad.numpy(), rtol=1e-12, atol=1e-13)


def test_silu_backward_matches_finite_differences():
    rng = np.random.default_rng(12)
    M, d, f = 3, 8, 12
    x = rng.standard_normal((M, d))
    wgT, wuT, wd = (rng.standard_normal((f, d)) / 2 for _ in range(3))
    dy = rng.standard_normal((M, d))
    b = oracle.ffn_bwd_dense_silu(x, wgT, wuT, wd, dy)
    h = 1e-6
    for gname, arr in {"dx": x, "dwgT": wgT, "dwuT": wuT, "dwd": wd}.items():
        for flat in range(arr.size):
            i = np.unravel_index(flat, arr.shape)
            old = arr[i]
            arr[i] = old + h
            lp = float((oracle.ffn_fwd_dense_silu(x, wgT, wuT, wd) * dy).sum())
            arr[i] = old - h
            lm = float((oracle.ffn_fwd_dense_silu(x, wgT, wuT, wd) * dy).sum())
            arr[i] = old
            fd = (lp - lm) / (2 * h)
            assert abs(fd - b[gname][i]) <= 1e-6 * max(1.0, abs(b[gname][i])), (gname, i)


def test_silu_equals_relu_when_every_gate_is_large():
    """sigmoid(a) = 1 to fp64 precision for a >= 40: SiLU and ReLU gates agree."""
    rng = np.random.default_rng(13)
    M, d, f = 5, 10, 16
    x = rng.standard_normal((M, d))
    x[:, -1] = 1.0
    wgT = rng.standard_normal((f, d)) / 4
    wgT[:, -1] = 60.0  # a = x . Wg >= 60 - |rest| > 40
    wuT, wd = rng.standard_normal((f, d)), rng.standard_normal((f, d))
    assert oracle.gate_preact(x, wgT).min() > 40
    np.testing.assert_allclose(oracle.ffn_fwd_dense_silu(x, wgT, wuT, wd),
                               oracle.ffn_fwd_dense(x, wgT, wuT, wd, round_g=False),
                               rtol=1e-13, atol=1e-12)
