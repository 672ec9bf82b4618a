"""The seeded generator produces the density it promises (binomial bounds)."""
import numpy as np

import oracle
from activation_sparse_gated_tcgen05_gb300 import synthetic


def test_bf16_bits_roundtrip():
    v = np.array([1.0, -2.5, 2.0 ** -130, 65280.0], np.float32)
    np.testing.assert_array_equal(synthetic.bf16_bits_to_f32(synthetic.to_bf16_bits(v)), v)


def test_seeded_and_reproducible():
    a = synthetic.make_inputs(8, 32, 64, seed=3)
    b = synthetic.make_inputs(8, 32, 64, seed=3)
    c = synthetic.make_inputs(8, 32, 64, seed=4)
    for k in ("x", "wgT", "wuT", "wd", "dy"):
        np.testing.assert_array_equal(a[k], b[k])
    assert (a["x"] != c["x"]).any()


def test_uniform_density_per_neuron_is_binomial():
    # For a fixed neuron the rows are independent draws, so its live count is
    # Binomial(M, p); the sum over neurons is checked against 5 binomial sigmas
    # (widened 1.5x for the weak coupling through shared rows).
    M, d, f, p = 16384, 256, 64, 0.005
    w = synthetic.make_inputs(M, d, f, density=p, seed=0, with_dy=False)
    live = oracle.gate_preact(w["x"], w["wgT"]) > 0
    n = live.sum()
    mean, sd = M * f * p, np.sqrt(M * f * p * (1 - p))
    assert abs(n - mean) < 5 * 1.5 * sd, (n, mean, sd)
    per_neuron = live.sum(0)
    sd1 = np.sqrt(M * p * (1 - p))
    assert np.abs(per_neuron - M * p).max() < 5 * sd1


def test_density_sweep_targets():
    M, d, f = 4096, 128, 128
    for p in synthetic.DENSITY_SWEEP:
        w = synthetic.make_inputs(M, d, f, density=p, seed=1, with_dy=False)
        frac = (oracle.gate_preact(w["x"], w["wgT"]) > 0).mean()
        sd = np.sqrt(p * (1 - p) / (M * f))
        assert abs(frac - p) < 6 * 1.5 * sd + 0.02 * p, (p, frac)


def test_lognormal_rows_follow_their_target():
    M, d, f = 2048, 128, 512
    w = synthetic.make_inputs(M, d, f, density=0.005, seed=2, lognormal_sigma=1.0,
                              with_dy=False)
    p = w["row_density"]
    assert p.max() <= 0.30 and abs(np.median(p) - 0.005) < 0.0015
    live = (oracle.gate_preact(w["x"], w["wgT"]) > 0).mean(1)
    # overall density matches the mean target; rows with a higher target are denser
    assert abs(live.mean() - p.mean()) < 0.1 * p.mean()
    order = np.argsort(p)
    lo, hi = live[order[: M // 4]].mean(), live[order[-M // 4:]].mean()
    assert hi > 5 * lo


def test_integer_gate_inputs_are_exact():
    w = synthetic.make_integer_gate_inputs(64, 256, 128, seed=0)
    x = synthetic.bf16_bits_to_f32(w["x"]).astype(np.float64)
    g = synthetic.bf16_bits_to_f32(w["wgT"]).astype(np.float64)
    assert (x == np.round(x)).all() and (g == np.round(g)).all()
    a = x @ g.T
    assert np.abs(a).max() < 2 ** 24
    assert 0.0005 < (a > 0).mean() < 0.03
