"""Seeded synthetic inputs for the activation-sparse gated FFN.

This module only draws inputs; it holds none of the FFN's arithmetic.  The
CUDA path and the CPU oracle are both fed from it, byte for byte.

Workload recipe (gated FFN of a Transformer++ with a ReLU gate whose output
is ~99.5 % exact zeros, page 2 "Sakana AI and NVIDIA introduce TwELL with CUDA
kernels ...", sections "¿Cuál es el problema que TwELL resuelve?" and
"Receta de entrenamiento"):

* x ~ N(0, 1) with the last feature held constant (the "constant feature");
* Wg, Wu ~ N(0, 1/d_model); Wd ~ N(0, 1/d_ff); dY ~ N(0, 1);
* the gate weight of the constant feature is set per neuron j to
  -z * ||Wg[0:d-1, j]||, z = Phi^-1(1 - p), so for x drawn as above
  P(a_mj > 0) = p for every neuron (a_mj = x_m . Wg[:, j]);
* per-row densities p_m (lognormal workloads) are obtained by setting the
  constant feature of row m to Phi^-1(1 - p_m) / z with z taken at p = 0.5 %.

All values are rounded to bf16 (round to nearest even) and returned as
uint16 bit patterns in the library's layouts: x, dy [M][d]; wgT, wuT, wd
[d_ff][d_model] (wgT / wuT are nn.Linear's weight layout, wd is Wd itself).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
from scipy.special import ndtri

DENSITY_REF = 0.005  # the pages' 99.5 % zeros


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def z_of_density(p):
    """z with P(N(0,1) > z) = p."""
    return ndtri(1.0 - np.asarray(p, dtype=np.float64))


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    d_model: int
    d_ff: int
    tile_n: int
    tile_cap: int
    density: float = DENSITY_REF          # uniform per-row target density
    lognormal_sigma: Optional[float] = None  # per-row lognormal density (median = density)
    density_cap: float = 0.30
    # ELL width W = the (1 - route_fraction) quantile of row_nnz; 0 means W = max row_nnz,
    # so only rows with an overflowing tile go to the dense backup
    route_fraction: float = 0.0
    seeds: tuple = (0,)


# The five workloads: tiny forward; 0.5B-class forward; 2B-class forward with a
# density sweep; 2B-class fwd+bwd with lognormal per-row density; 8B-class
# fwd+bwd with lognormal density (plus a small-M forward at that shape).
WORKLOADS = {
    "tiny_fwd": Workload("tiny_fwd", 256, 256, 1024, 64, 16),
    "fwd_0p5b": Workload("fwd_0p5b", 16384, 1024, 4096, 128, 32, seeds=(0, 1, 2)),
    "fwd_2b": Workload("fwd_2b", 32768, 2048, 8192, 128, 32),
    "train_2b": Workload("train_2b", 16384, 2048, 8192, 128, 32, lognormal_sigma=1.0,
                         route_fraction=0.03),
    "train_8b": Workload("train_8b", 16384, 4096, 14336, 128, 32, lognormal_sigma=0.7,
                         route_fraction=0.03),
}
DENSITY_SWEEP = (0.0025, 0.005, 0.01, 0.02, 0.05)
SMALL_M = (1, 16, 64)


def ell_width(row_nnz: np.ndarray, route_fraction: float) -> int:
    """ELL width that sends about `route_fraction` of the rows to the dense
    backup (0: the widest row, so none is routed for its length)."""
    nnz = np.sort(np.asarray(row_nnz).reshape(-1))
    if nnz.size == 0:
        return 0
    if route_fraction <= 0:
        return int(nnz[-1])
    return int(nnz[min(nnz.size - 1, int((1.0 - route_fraction) * nnz.size))])


def row_densities(M: int, median: float, sigma: Optional[float], cap: float,
                  rng: np.random.Generator) -> np.ndarray:
    if sigma is None:
        return np.full(M, median, dtype=np.float64)
    z = rng.standard_normal(M)
    return np.minimum(cap, median * np.exp(sigma * z))


def make_inputs(M: int, d: int, f: int, density: float = DENSITY_REF, seed: int = 0,
                lognormal_sigma: Optional[float] = None, density_cap: float = 0.30,
                with_dy: bool = True) -> dict:
    """Draw one workload.  Returns a dict of bf16 bit arrays (uint16) plus
    ``row_density`` (the per-row target p_m, float64)."""
    if d < 2:
        raise ValueError("d_model must be >= 2 (the last feature is the constant one)")
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((M, d), dtype=np.float32)
    wg = rng.standard_normal((f, d), dtype=np.float32) * np.float32(1.0 / np.sqrt(d))
    wu = rng.standard_normal((f, d), dtype=np.float32) * np.float32(1.0 / np.sqrt(d))
    wd = rng.standard_normal((f, d), dtype=np.float32) * np.float32(1.0 / np.sqrt(f))
    dy = rng.standard_normal((M, d), dtype=np.float32) if with_dy else None
    p_row = row_densities(M, density, lognormal_sigma, density_cap, rng)

    if lognormal_sigma is None:
        z_ref = float(z_of_density(density))
        x[:, d - 1] = 1.0
    else:
        z_ref = float(z_of_density(density))
        x[:, d - 1] = (z_of_density(p_row) / z_ref).astype(np.float32)

    wg_bits = to_bf16_bits(wg)
    body = bf16_bits_to_f32(wg_bits[:, : d - 1]).astype(np.float64)
    norm = np.sqrt(np.einsum("jk,jk->j", body, body))
    wg_bits[:, d - 1] = to_bf16_bits((-z_ref * norm).astype(np.float32))

    out = {
        "x": to_bf16_bits(x),
        "wgT": wg_bits,
        "wuT": to_bf16_bits(wu),
        "wd": to_bf16_bits(wd),
        "row_density": p_row,
    }
    if with_dy:
        out["dy"] = to_bf16_bits(dy)
    return out


def make_workload(w: Workload, seed: Optional[int] = None, M: Optional[int] = None,
                  density: Optional[float] = None, with_dy: bool = True) -> dict:
    return make_inputs(M if M is not None else w.M, w.d_model, w.d_ff,
                       density=w.density if density is None else density,
                       seed=w.seeds[0] if seed is None else seed,
                       lognormal_sigma=w.lognormal_sigma, density_cap=w.density_cap,
                       with_dy=with_dy)


def make_integer_gate_inputs(M: int, d: int, f: int, density: float = DENSITY_REF,
                             seed: int = 0, mixed_rows: bool = False) -> dict:
    """Gate inputs whose products and partial sums are small integers, so any
    summation order in fp32 gives the same exact pre-activation.  x in
    {-2..2}, Wg in {-3..3}, constant last feature 1 with a per-neuron integer
    offset chosen for density ``density``.  Every value is exact in bf16.

    With ``mixed_rows`` the constant feature of each row is drawn from
    {0, 1, 2} with probabilities (0.05, 0.9, 0.05): rows at ~50 %, at
    ``density`` and at almost 0 % density, a non-uniform mix that exercises
    the hybrid routing."""
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    x = rng.integers(-2, 3, size=(M, d)).astype(np.float32)
    wg = rng.integers(-3, 4, size=(f, d)).astype(np.float32)
    x[:, d - 1] = 1.0
    if mixed_rows:
        x[:, d - 1] = rng.choice(np.array([0.0, 1.0, 2.0], np.float32), size=M,
                                 p=[0.05, 0.9, 0.05])
    sd = np.sqrt((d - 1) * 2.0 * 4.0)  # Var(x) = 2, Var(w) = 4
    off = np.round(float(z_of_density(density)) * sd)
    # keep the offset exactly representable in bf16 (8 significant bits)
    off_bits = to_bf16_bits(np.float32(-off))
    wg_bits = to_bf16_bits(wg)
    wg_bits[:, d - 1] = off_bits
    return {"x": to_bf16_bits(x), "wgT": wg_bits}


def make_exact_gate_inputs(M: int, d: int, f: int, density: float = DENSITY_REF,
                           seed: int = 0, mixed_rows: bool = False) -> dict:
    """A full FFN workload whose gate pre-activation is exact in fp32 (see
    make_integer_gate_inputs), with Wu, Wd, dY drawn as in make_inputs."""
    out = make_integer_gate_inputs(M, d, f, density, seed, mixed_rows)
    rng = np.random.Generator(np.random.PCG64(seed + 3000))
    out["wuT"] = to_bf16_bits(rng.standard_normal((f, d), dtype=np.float32)
                              * np.float32(1.0 / np.sqrt(d)))
    out["wd"] = to_bf16_bits(rng.standard_normal((f, d), dtype=np.float32)
                             * np.float32(1.0 / np.sqrt(f)))
    out["dy"] = to_bf16_bits(rng.standard_normal((M, d), dtype=np.float32))
    return out


def make_sparse_preact(M: int, f: int, density: float, seed: int = 0,
                       dtype=np.float32) -> np.ndarray:
    """A dense pre-activation matrix with P(a > 0) = density: N(0,1) values
    shifted down by z(density).  Used to drive the pack-from-dense path with
    identical bytes on both sides.  A few special values are planted: -0.0,
    +0.0, tiny positives that round to zero in bf16, NaN and +inf."""
    rng = np.random.Generator(np.random.PCG64(seed + 2000))
    a = (rng.standard_normal((M, f)) - z_of_density(density)).astype(dtype)
    if M * f >= 8:
        flat = a.reshape(-1)
        pos = rng.choice(M * f, size=8, replace=False)
        specials = np.array([-0.0, 0.0, 1e-45, -1e-45, np.nan, np.inf, -np.inf, 3e-39],
                            dtype=np.float64)
        flat[pos] = specials.astype(dtype)
    return a
