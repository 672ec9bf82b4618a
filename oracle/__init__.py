"""CPU oracle for the activation-sparse gated FFN (TwELL) -- test infrastructure.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``twell_oracle.cpp`` (plain
fp64 loops, see that file for the definitions and the pages they follow)
through ctypes, and shares nothing with the CUDA library: it has its own
bf16 decoding, its own packer, router and forward/backward statements.

Arrays passed in may be bf16 bit patterns (``uint16``), float32 or float64;
they are decoded exactly to float64 before the C code sees them.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_U16 = ctypes.POINTER(ctypes.c_uint16)
_U8 = ctypes.POINTER(ctypes.c_uint8)
_I32 = ctypes.POINTER(ctypes.c_int32)
_I64 = ctypes.POINTER(ctypes.c_int64)
_i64 = ctypes.c_int64
_int = ctypes.c_int


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = _build.OUT
    if not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_build.SRC):
        _build.build()
    lib = ctypes.CDLL(path)
    sig = {
        "orc_set_threads": (None, [_int]),
        "orc_get_threads": (_int, []),
        "orc_double_to_bf16": (None, [_D, _i64, _U16]),
        "orc_gate_preact": (None, [_D, _D, _i64, _i64, _i64, _D]),
        "orc_twell_pack": (None, [_D, _i64, _i64, _int, _int, _U16, _U8, _U8, _I32]),
        "orc_twell_unpack": (None, [_U16, _U8, _U8, _i64, _i64, _int, _int, _D]),
        "orc_hybrid_route": (None, [_U16, _U8, _U8, _I32, _i64, _i64, _int, _int, ctypes.c_int32,
                                    _U16, _U16, _I32, _I32, _I32]),
        "orc_ffn_fwd_dense": (None, [_D, _D, _D, _D, _i64, _i64, _int, _I64, _i64, _D]),
        "orc_ffn_fwd_dense_silu": (None, [_D, _D, _D, _D, _i64, _i64, _I64, _i64, _D]),
        "orc_ffn_bwd_dense_silu": (None, [_D, _D, _D, _D, _D, _i64, _i64, _i64, _D, _D, _D,
                                          _D]),
        "orc_ffn_fwd_twell": (None, [_D, _D, _D, _i64, _i64, _int, _int, _U16, _U8, _U8,
                                     _I64, _i64, _D]),
        "orc_ffn_fwd_ell": (None, [_D, _D, _D, _i64, ctypes.c_int32, _U16, _U16, _I32, _I64,
                                   _i64, _D]),
        "orc_ffn_bwd_dense": (None, [_D, _D, _D, _D, _D, _i64, _i64, _i64, ctypes.c_double, _int,
                                     _D, _D, _D, _D, _D]),
        "orc_ffn_bwd_dx_rows": (None, [_D, _D, _D, _D, _D, _i64, _i64, ctypes.c_double, _int,
                                       _I64, _i64, _D]),
        "orc_ffn_bwd_dw_neurons": (None, [_D, _D, _D, _D, _D, _i64, _i64, ctypes.c_double, _int,
                                          _I64, _i64, _D, _D, _D]),
        "orc_ffn_bwd_hybrid": (None, [_D, _D, _D, _D, _D, _i64, _i64, _i64, ctypes.c_int32, _U16,
                                      _U16, _I32, _I32, ctypes.c_int32, ctypes.c_double,
                                      _D, _D, _D, _D]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def set_threads(n: int) -> None:
    """Number of host threads the oracle may use (results do not depend on it)."""
    _load().orc_set_threads(int(n))


def get_threads() -> int:
    return int(_load().orc_get_threads())


# ---------------------------------------------------------------- conversions
def f64(a) -> np.ndarray:
    """Decode an array to contiguous float64; uint16 is read as bf16 bits."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a, typ):
    return a.ctypes.data_as(typ)


def double_to_bf16(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().orc_double_to_bf16(_p(v, _D), v.size, _p(out, _U16))
    return out


# ---------------------------------------------------------------- forward
def gate_preact(x, wgT) -> np.ndarray:
    """a = x Wg in fp64; x [M][d], wgT [f][d] -> [M][f]."""
    x, w = f64(x), f64(wgT)
    M, d = x.shape
    f = w.shape[0]
    a = np.empty((M, f), np.float64)
    _load().orc_gate_preact(_p(x, _D), _p(w, _D), M, d, f, _p(a, _D))
    return a


def twell_pack(a, tile_n: int, cap: int):
    """Naive TwELL packer.  Returns (val bf16-bits [M][T][C], idx u8, cnt u8 [M][T],
    row_nnz i32 [M]); slots at or past min(cnt, C) are zero."""
    a = f64(a)
    M, f = a.shape
    T = f // tile_n
    val = np.zeros((M, T, cap), np.uint16)
    idx = np.zeros((M, T, cap), np.uint8)
    cnt = np.zeros((M, T), np.uint8)
    nnz = np.zeros(M, np.int32)
    _load().orc_twell_pack(_p(a, _D), M, f, tile_n, cap, _p(val, _U16), _p(idx, _U8),
                           _p(cnt, _U8), _p(nnz, _I32))
    return val, idx, cnt, nnz


def twell_unpack(val, idx, cnt, f: int, tile_n: int) -> np.ndarray:
    val = np.ascontiguousarray(val, np.uint16)
    idx = np.ascontiguousarray(idx, np.uint8)
    cnt = np.ascontiguousarray(cnt, np.uint8)
    M, T, C = val.shape
    g = np.empty((M, f), np.float64)
    _load().orc_twell_unpack(_p(val, _U16), _p(idx, _U8), _p(cnt, _U8), M, f, tile_n, C, _p(g, _D))
    return g


def hybrid_route(val, idx, cnt, row_nnz, f: int, tile_n: int, ell_width: int):
    """Returns (ell_val bf16-bits [M][W], ell_col u16 [M][W], ell_nnz i32 [M],
    dense_rows i32 [n_dense]); unused ELL slots are zero."""
    val = np.ascontiguousarray(val, np.uint16)
    idx = np.ascontiguousarray(idx, np.uint8)
    cnt = np.ascontiguousarray(cnt, np.uint8)
    row_nnz = np.ascontiguousarray(row_nnz, np.int32)
    M, T, C = val.shape
    W = int(ell_width)
    ev = np.zeros((M, max(W, 1)), np.uint16)
    ec = np.zeros((M, max(W, 1)), np.uint16)
    en = np.zeros(M, np.int32)
    dr = np.zeros(M, np.int32)
    nd = np.zeros(1, np.int32)
    _load().orc_hybrid_route(_p(val, _U16), _p(idx, _U8), _p(cnt, _U8), _p(row_nnz, _I32), M, f,
                             tile_n, C, W, _p(ev, _U16), _p(ec, _U16), _p(en, _I32), _p(dr, _I32),
                             _p(nd, _I32))
    return ev[:, :W], ec[:, :W], en, dr[: int(nd[0])].copy()


def _rows(rows, M):
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    return np.ascontiguousarray(rows, dtype=np.int64)


def ffn_fwd_dense(x, wgT, wuT, wd, rows=None, round_g: bool = True) -> np.ndarray:
    """y = (ReLU(x Wg) * (x Wu)) Wd in fp64 for the listed rows ([len(rows)][d])."""
    x, wg, wu, wdd = f64(x), f64(wgT), f64(wuT), f64(wd)
    M, d = x.shape
    f = wg.shape[0]
    r = _rows(rows, M)
    y = np.empty((r.size, d), np.float64)
    _load().orc_ffn_fwd_dense(_p(x, _D), _p(wg, _D), _p(wu, _D), _p(wdd, _D), d, f,
                              int(round_g), _p(r, _I64), r.size, _p(y, _D))
    return y


def ffn_fwd_dense_silu(x, wgT, wuT, wd, rows=None) -> np.ndarray:
    """y = (SiLU(x Wg) * (x Wu)) Wd in fp64 (the unmodified gated FFN)."""
    x, wg, wu, wdd = f64(x), f64(wgT), f64(wuT), f64(wd)
    M, d = x.shape
    f = wg.shape[0]
    r = _rows(rows, M)
    y = np.empty((r.size, d), np.float64)
    _load().orc_ffn_fwd_dense_silu(_p(x, _D), _p(wg, _D), _p(wu, _D), _p(wdd, _D), d, f,
                                   _p(r, _I64), r.size, _p(y, _D))
    return y


def ffn_bwd_dense_silu(x, wgT, wuT, wd, dy):
    """Whole-batch backward of the SiLU-gated FFN (no L1 term; small shapes).
    Returns dict dx, dwgT, dwuT, dwd."""
    x, wg, wu, wdd, dyy = f64(x), f64(wgT), f64(wuT), f64(wd), f64(dy)
    M, d = x.shape
    f = wg.shape[0]
    dx = np.empty((M, d))
    dwg = np.empty((f, d))
    dwu = np.empty((f, d))
    dwd = np.empty((f, d))
    _load().orc_ffn_bwd_dense_silu(_p(x, _D), _p(wg, _D), _p(wu, _D), _p(wdd, _D), _p(dyy, _D),
                                   M, d, f, _p(dx, _D), _p(dwg, _D), _p(dwu, _D), _p(dwd, _D))
    return {"dx": dx, "dwgT": dwg, "dwuT": dwu, "dwd": dwd}


def ffn_fwd_twell(x, wuT, wd, val, idx, cnt, tile_n: int, rows=None) -> np.ndarray:
    """y from the stored TwELL entries only (fp64)."""
    x, wu, wdd = f64(x), f64(wuT), f64(wd)
    val = np.ascontiguousarray(val, np.uint16)
    idx = np.ascontiguousarray(idx, np.uint8)
    cnt = np.ascontiguousarray(cnt, np.uint8)
    M, d = x.shape
    f = wu.shape[0]
    C = val.shape[2]
    r = _rows(rows, M)
    y = np.empty((r.size, d), np.float64)
    _load().orc_ffn_fwd_twell(_p(x, _D), _p(wu, _D), _p(wdd, _D), d, f, tile_n, C,
                              _p(val, _U16), _p(idx, _U8), _p(cnt, _U8), _p(r, _I64), r.size,
                              _p(y, _D))
    return y


def ffn_fwd_ell(x, wuT, wd, ell_val, ell_col, ell_nnz, rows=None) -> np.ndarray:
    """y from the stored ELL entries only (fp64); routed rows (ell_nnz = 0) give 0."""
    x, wu, wdd = f64(x), f64(wuT), f64(wd)
    ev = np.ascontiguousarray(ell_val, np.uint16)
    ec = np.ascontiguousarray(ell_col, np.uint16)
    en = np.ascontiguousarray(ell_nnz, np.int32)
    M, d = x.shape
    W = ev.shape[1]
    if W == 0:
        ev = np.zeros((M, 1), np.uint16)
        ec = np.zeros((M, 1), np.uint16)
    r = _rows(rows, M)
    y = np.empty((r.size, d), np.float64)
    _load().orc_ffn_fwd_ell(_p(x, _D), _p(wu, _D), _p(wdd, _D), d, max(W, 1) if W == 0 else W,
                            _p(ev, _U16), _p(ec, _U16), _p(en, _I32), _p(r, _I64), r.size,
                            _p(y, _D))
    return y


def ffn_bwd_dense(x, wgT, wuT, wd, dy, l1_coeff: float, round_g: bool = True):
    """Whole-batch backward (small shapes).  Returns dict dx, dwgT, dwuT, dwd, l1."""
    x, wg, wu, wdd, dyy = f64(x), f64(wgT), f64(wuT), f64(wd), f64(dy)
    M, d = x.shape
    f = wg.shape[0]
    dx = np.empty((M, d))
    dwg = np.empty((f, d))
    dwu = np.empty((f, d))
    dwd = np.empty((f, d))
    l1 = np.zeros(1)
    _load().orc_ffn_bwd_dense(_p(x, _D), _p(wg, _D), _p(wu, _D), _p(wdd, _D), _p(dyy, _D), M, d,
                              f, float(l1_coeff), int(round_g), _p(dx, _D), _p(dwg, _D),
                              _p(dwu, _D), _p(dwd, _D), _p(l1, _D))
    return {"dx": dx, "dwgT": dwg, "dwuT": dwu, "dwd": dwd, "l1": float(l1[0])}


def ffn_bwd_dx_rows(x, wgT, wuT, wd, dy, l1_coeff: float, rows, round_g: bool = True):
    x, wg, wu, wdd, dyy = f64(x), f64(wgT), f64(wuT), f64(wd), f64(dy)
    M, d = x.shape
    f = wg.shape[0]
    r = _rows(rows, M)
    dx = np.empty((r.size, d))
    _load().orc_ffn_bwd_dx_rows(_p(x, _D), _p(wg, _D), _p(wu, _D), _p(wdd, _D), _p(dyy, _D), d, f,
                                float(l1_coeff), int(round_g), _p(r, _I64), r.size, _p(dx, _D))
    return dx


def ffn_bwd_dw_neurons(x, wgT, wuT, wd, dy, l1_coeff: float, neurons, round_g: bool = True):
    """(dwgT, dwuT, dwd) rows for the listed neurons, each [len(neurons)][d]."""
    x, wg, wu, wdd, dyy = f64(x), f64(wgT), f64(wuT), f64(wd), f64(dy)
    M, d = x.shape
    n = np.ascontiguousarray(neurons, dtype=np.int64)
    og = np.empty((n.size, d))
    ou = np.empty((n.size, d))
    od = np.empty((n.size, d))
    _load().orc_ffn_bwd_dw_neurons(_p(x, _D), _p(wg, _D), _p(wu, _D), _p(wdd, _D), _p(dyy, _D),
                                   M, d, float(l1_coeff), int(round_g), _p(n, _I64), n.size,
                                   _p(og, _D), _p(ou, _D), _p(od, _D))
    return og, ou, od


def ffn_bwd_hybrid(x, wgT, wuT, wd, dy, ell_val, ell_col, ell_nnz, dense_rows, l1_coeff: float):
    """Backward that walks the hybrid format: ELL rows over stored entries,
    routed rows by the dense definitions.  Returns dict dx, dwgT, dwuT, dwd."""
    x, wg, wu, wdd, dyy = f64(x), f64(wgT), f64(wuT), f64(wd), f64(dy)
    M, d = x.shape
    f = wg.shape[0]
    ev = np.ascontiguousarray(ell_val, np.uint16)
    ec = np.ascontiguousarray(ell_col, np.uint16)
    W = ev.shape[1]
    if W == 0:
        ev = np.zeros((M, 1), np.uint16)
        ec = np.zeros((M, 1), np.uint16)
    en = np.ascontiguousarray(ell_nnz, np.int32)
    dr = np.ascontiguousarray(dense_rows, np.int32)
    if dr.size == 0:
        dr_buf = np.zeros(1, np.int32)
    else:
        dr_buf = dr
    dx = np.empty((M, d))
    dwg = np.empty((f, d))
    dwu = np.empty((f, d))
    dwd = np.empty((f, d))
    _load().orc_ffn_bwd_hybrid(_p(x, _D), _p(wg, _D), _p(wu, _D), _p(wdd, _D), _p(dyy, _D), M, d,
                               f, max(W, 1) if W == 0 else W, _p(ev, _U16), _p(ec, _U16),
                               _p(en, _I32), _p(dr_buf, _I32), int(dr.size), float(l1_coeff),
                               _p(dx, _D), _p(dwg, _D), _p(dwu, _D), _p(dwd, _D))
    return {"dx": dx, "dwgT": dwg, "dwuT": dwu, "dwd": dwd}
