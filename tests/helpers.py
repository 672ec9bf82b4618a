"""Shared test helpers: device upload of the generator's bf16 bits and the
float tolerance of the parity tests.

Float tolerance (bf16 inputs, fp32 accumulation): relative Frobenius error
<= 5e-3 and max |error| <= 2e-2 * rms(reference).  An output stored as bf16
(y, dx) also carries its own storage rounding, up to 2^-8 * |reference| per
element (round to nearest, 8 significant bits); that term is added to the
max-|error| bound for bf16 outputs, since no bf16 result can avoid it."""
import numpy as np
import torch

REL_FRO = 5e-3
MAX_ABS_RMS = 2e-2


def dev_bf16(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def assert_close(got, ref, name="", rel=REL_FRO, max_rms=MAX_ABS_RMS, out_bf16=False,
                 allowance=None):
    """Tolerance check.  `allowance` (same shape as ref) widens the per-element
    bound by the effect of gate rounding decisions that may go either way
    (see gate_decisions); the Frobenius criterion is applied to the error
    left after removing that part."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), name + ": non-finite output"
    nr = np.linalg.norm(ref)
    diff = got - ref
    if allowance is not None:
        diff = np.sign(diff) * np.maximum(np.abs(diff) - allowance, 0.0)
    err = np.linalg.norm(diff)
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    if nr == 0.0:
        assert err == 0.0, "%s: expected exact zeros, |err| = %g" % (name, err)
        return
    assert err / nr <= rel, "%s: relative Frobenius error %.3g > %.3g" % (name, err / nr, rel)
    bound = max_rms * rms + (2.0 ** -8 * np.abs(ref) if out_bf16 else 0.0)
    excess = np.abs(diff) - bound
    k = int(np.argmax(excess))
    assert excess.flat[k] <= 0, "%s: |err| %.3g at %d exceeds bound %.3g (rms %.3g, ref %.3g)" % (
        name, np.abs(diff).flat[k], k, np.broadcast_to(bound, ref.shape).flat[k], rms,
        ref.flat[k])


def gate_decisions(w, rows=None):
    """Where the gate's rounding decisions may legitimately differ.

    g = bf16(ReLU(a)) is decided on the kernel's fp32 pre-activation, whose
    accumulation error is at most d * 2^-23 * sum_k |x_k w_k|.  Inside that
    band around the fp64 a, the stored g may be either neighbouring bf16
    value (dg = their difference) and, near zero, the entry may be live or
    dead (flip).  Returns (a, dg, flip) for the given rows, from the oracle."""
    import oracle

    x = oracle.f64(w["x"])
    if rows is not None:
        x = x[rows]
    wg = oracle.f64(w["wgT"])
    a = oracle.gate_preact(x, wg)
    band = x.shape[1] * 2.0 ** -23 * (np.abs(x) @ np.abs(wg).T)
    g_lo = oracle.f64(oracle.double_to_bf16(np.maximum(a - band, 0.0)))
    g_hi = oracle.f64(oracle.double_to_bf16(np.maximum(a + band, 0.0)))
    flip = (a - band <= 0.0) & (a + band > 0.0)
    return a, g_hi - g_lo, flip


def fwd_allowance(w, rows=None):
    """Bound on |dy| caused by the gate decisions of gate_decisions()."""
    import oracle

    x = oracle.f64(w["x"])
    if rows is not None:
        x = x[rows]
    _, dg, _ = gate_decisions(w, rows)
    u = x @ oracle.f64(w["wuT"]).T
    return (dg * np.abs(u)) @ np.abs(oracle.f64(w["wd"]))


def bwd_allowance(w, lam):
    """Bounds on |d dx|, |d dWg^T|, |d dWu^T|, |d dWd| caused by the gate
    decisions (whole batch; small shapes)."""
    import oracle

    x, dy = oracle.f64(w["x"]), oracle.f64(w["dy"])
    wg, wu, wd = oracle.f64(w["wgT"]), oracle.f64(w["wuT"]), oracle.f64(w["wd"])
    _, dg, flip = gate_decisions(w)
    u = x @ wu.T
    dh = dy @ wd.T
    da_mag = np.where(flip, np.abs(dh * u + lam), 0.0)
    return {
        "dx": (np.abs(dh) * dg) @ np.abs(wu) + da_mag @ np.abs(wg),
        "dwgT": da_mag.T @ np.abs(x),
        "dwuT": (np.abs(dh) * dg).T @ np.abs(x),
        "dwd": (dg * np.abs(u)).T @ np.abs(dy),
    }


def dense_intermediate_allowance(w, lam):
    """Bounds for a dense bf16 FFN that stores its intermediates h, u, du, da
    as bf16 between GEMMs (the library's dense comparator): each stored value
    carries a relative rounding error of at most 2^-8, which first-order
    propagates as 2^-8 * (|terms| @ |weights|) into each output."""
    import oracle

    x, dy = oracle.f64(w["x"]), oracle.f64(w["dy"])
    wg, wu, wd = oracle.f64(w["wgT"]), oracle.f64(w["wuT"]), oracle.f64(w["wd"])
    a = x @ wg.T
    g = oracle.f64(oracle.double_to_bf16(np.maximum(a, 0.0)))
    u = x @ wu.T
    h = g * u
    dh = dy @ wd.T
    du = dh * g
    da_err = np.where(g > 0, np.abs(dh * u + lam) + np.abs(dh * u), 0.0)  # da and u both stored
    r = 2.0 ** -8
    return {
        "y": r * np.abs(h) @ np.abs(wd),
        "dx": r * (np.abs(du) @ np.abs(wu) + da_err @ np.abs(wg)),
        "dwgT": r * da_err.T @ np.abs(x),
        "dwuT": r * np.abs(du).T @ np.abs(x),
        "dwd": r * np.abs(h).T @ np.abs(dy),
    }


def dense_silu_intermediate_allowance(w):
    """dense_intermediate_allowance for the SiLU-gated comparator, which keeps
    bf16(a), u, h, du, da between its GEMMs.  Each stored value carries a
    relative rounding error of at most 2^-8; the backward recomputes
    s = silu(a) and s'(a) from the rounded a, so a's error enters du through
    s'(a) and da through s''(a).  First order, propagated through |weights|."""
    import oracle

    x, dy = oracle.f64(w["x"]), oracle.f64(w["dy"])
    wg, wu, wd = oracle.f64(w["wgT"]), oracle.f64(w["wuT"]), oracle.f64(w["wd"])
    a = x @ wg.T
    sg = 1.0 / (1.0 + np.exp(-a))
    s = a * sg
    ds = sg * (1.0 + a * (1.0 - sg))
    d2s = sg * (1.0 - sg) * (2.0 + a * (1.0 - 2.0 * sg))
    u = x @ wu.T
    h = s * u
    dh = dy @ wd.T
    du = dh * s
    da = dh * u * ds
    r = 2.0 ** -8
    du_err = r * (np.abs(du) + np.abs(dh * ds * a))
    da_err = r * (np.abs(da) + np.abs(dh * u * d2s * a) + np.abs(dh * ds * u))
    return {
        "y": r * np.abs(h) @ np.abs(wd),
        "dx": du_err @ np.abs(wu) + da_err @ np.abs(wg),
        "dwgT": da_err.T @ np.abs(x),
        "dwuT": du_err.T @ np.abs(x),
        "dwd": r * np.abs(h).T @ np.abs(dy),
    }


def bwd_allowance_sampled(w, lam, rows, neurons):
    """bwd_allowance restricted to dX of `rows` and dW of `neurons` (so it
    scales to full-size workloads)."""
    import oracle

    x, dy = oracle.f64(w["x"]), oracle.f64(w["dy"])
    wg, wu, wd = oracle.f64(w["wgT"]), oracle.f64(w["wuT"]), oracle.f64(w["wd"])
    d = x.shape[1]

    def decisions(xs, wgs):
        a = xs @ wgs.T
        band = d * 2.0 ** -23 * (np.abs(xs) @ np.abs(wgs).T)
        g_lo = oracle.f64(oracle.double_to_bf16(np.maximum(a - band, 0.0)))
        g_hi = oracle.f64(oracle.double_to_bf16(np.maximum(a + band, 0.0)))
        return g_hi - g_lo, (a - band <= 0.0) & (a + band > 0.0)

    out = {}
    xr = x[rows]
    dg, flip = decisions(xr, wg)
    u = xr @ wu.T
    dh = dy[rows] @ wd.T
    out["dx"] = (np.abs(dh) * dg) @ np.abs(wu) + np.where(flip, np.abs(dh * u + lam), 0.0) @ np.abs(wg)
    dg, flip = decisions(x, wg[neurons])        # [M][n]
    u = x @ wu[neurons].T
    dh = dy @ wd[neurons].T
    out["dwgT"] = np.where(flip, np.abs(dh * u + lam), 0.0).T @ np.abs(x)
    out["dwuT"] = (np.abs(dh) * dg).T @ np.abs(x)
    out["dwd"] = (dg * np.abs(u)).T @ np.abs(dy)
    return out
