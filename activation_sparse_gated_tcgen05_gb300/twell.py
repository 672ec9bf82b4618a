"""Thin ctypes binding of libtwell.so (the C ABI in include/twell.h).

Argument marshalling only: every step of the FFN runs in the library's CUDA
kernels.  Functions carry the C names and take torch tensors that already
live on the GPU; they pass raw device pointers and the current CUDA stream.
A non-zero status raises TwellError.  There is no fallback: if the library
is missing or a call fails, the call raises.

Helpers ``alloc_tiles`` / ``alloc_hybrid`` allocate the packed-format
buffers with torch (device memory is the caller's in the C ABI).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

from . import _build

_lib = None

STATUS = {
    0: "TWELL_OK", 1: "TWELL_ERR_INVALID_ARG", 2: "TWELL_ERR_UNSUPPORTED",
    3: "TWELL_ERR_ALIGNMENT", 4: "TWELL_ERR_CAPACITY", 5: "TWELL_ERR_CUDA",
    6: "TWELL_ERR_DEVICE_TIMEOUT", 7: "TWELL_ERR_WORKSPACE", 8: "TWELL_ERR_INDEX",
}
EXPORTS = (
    "twell_pack", "twell_pack_dense", "hybrid_route", "twell_workspace_bytes",
    "twell_workspace_bytes_capped",
    "twell_tiles_workspace_bytes", "twell_set_split_gathers", "twell_set_pair_gemm",
    "twell_ffn_fwd",
    "twell_ffn_bwd", "twell_dense_workspace_bytes", "twell_dense_ffn_fwd", "twell_dense_ffn_bwd",
    "twell_dense_ffn_fwd_act", "twell_dense_ffn_bwd_act",
    "twell_gemm_bf16", "twell_get_device_status", "twell_status_string", "twell_num_sms",
    "twell_launch_count", "twell_profile_begin", "twell_profile_end", "twell_profile_entry",
    "twell_ffn_fwd_noalloc", "twell_selftest_wait_timeout",
)


class TwellError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__("%s failed: %s (%d)" % (fn, STATUS.get(status, "?"), status))
        self.status = status


class Shape(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int32), ("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("tile_n", ctypes.c_int32), ("tile_cap", ctypes.c_int32)]


class Tiles(ctypes.Structure):
    _fields_ = [("val", ctypes.c_void_p), ("idx", ctypes.c_void_p), ("cnt", ctypes.c_void_p),
                ("row_nnz", ctypes.c_void_p)]


class Hybrid(ctypes.Structure):
    _fields_ = [("ell_val", ctypes.c_void_p), ("ell_col", ctypes.c_void_p),
                ("ell_nnz", ctypes.c_void_p), ("ell_width", ctypes.c_int32),
                ("dense_rows", ctypes.c_void_p), ("n_dense", ctypes.c_void_p),
                ("dense_cap", ctypes.c_int32)]


def library_path() -> str:
    """libtwell.so, or the checked (bounds-checking debug) build
    libtwell_checked.so when the environment sets TWELL_CHECKED=1."""
    return _build.CHECKED_LIB if os.environ.get("TWELL_CHECKED") == "1" else _build.LIB


def load():
    """Load the library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError("libtwell.so not found at %s: run __graft_entry__.build() "
                           "(or python -m activation_sparse_gated_tcgen05_gb300._build)" % path)
    lib = ctypes.CDLL(path)
    P, I32, SZ, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    SP, TP, HP = ctypes.POINTER(Shape), ctypes.POINTER(Tiles), ctypes.POINTER(Hybrid)
    sig = {
        "twell_pack": (I32, [P, P, SP, TP, P]),
        "twell_pack_dense": (I32, [P, I32, SP, TP, P]),
        "hybrid_route": (I32, [TP, SP, HP, P]),
        "twell_workspace_bytes": (SZ, [SP, I32, I32]),
        "twell_workspace_bytes_capped": (SZ, [SP, I32, I32, I32]),
        "twell_tiles_workspace_bytes": (SZ, [SP]),
        "twell_set_split_gathers": (I32, [I32]),
        "twell_set_pair_gemm": (I32, [I32]),
        "twell_ffn_fwd": (I32, [P, P, P, P, SP, TP, HP, P, P, SZ, P]),
        "twell_ffn_bwd": (I32, [P, P, P, P, P, SP, HP, F, P, P, P, P, P, SZ, P]),
        "twell_ffn_fwd_noalloc": (I32, [P, P, P, P, SP, HP, P, P]),
        "twell_selftest_wait_timeout": (I32, [I32, P]),
        "twell_dense_workspace_bytes": (SZ, [SP, I32]),
        "twell_dense_ffn_fwd": (I32, [P, P, P, P, SP, P, I32, P, SZ, P]),
        "twell_dense_ffn_bwd": (I32, [P, P, P, P, P, SP, F, P, P, P, P, P, SZ, P]),
        "twell_dense_ffn_fwd_act": (I32, [P, P, P, P, SP, I32, P, I32, P, SZ, P]),
        "twell_dense_ffn_bwd_act": (I32, [P, P, P, P, P, SP, I32, F, P, P, P, P, P, SZ, P]),
        "twell_gemm_bf16": (I32, [P, P, P, I32, I32, I32, I32, I32, I32, I32, P]),
        "twell_get_device_status": (I32, [P, ctypes.POINTER(I32)]),
        "twell_status_string": (ctypes.c_char_p, [I32]),
        "twell_num_sms": (I32, []),
        "twell_launch_count": (ctypes.c_uint64, []),
        "twell_profile_begin": (I32, [ctypes.c_char_p]),
        "twell_profile_end": (I32, []),
        "twell_profile_entry": (I32, [I32, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(I32),
                                      ctypes.POINTER(ctypes.c_double)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(name: str, status: int):
    if status != 0:
        raise TwellError(name, status)


@dataclass
class TwellTiles:
    val: torch.Tensor      # bf16 [M][T][C]
    idx: torch.Tensor      # uint8 [M][T][C]
    cnt: torch.Tensor      # uint8 [M][T]
    row_nnz: torch.Tensor  # int32 [M]

    def c(self) -> Tiles:
        return Tiles(_ptr(self.val), _ptr(self.idx), _ptr(self.cnt), _ptr(self.row_nnz))


@dataclass
class TwellHybrid:
    ell_val: torch.Tensor     # bf16 [M][W]
    ell_col: torch.Tensor     # uint16 stored as int16 [M][W]
    ell_nnz: torch.Tensor     # int32 [M]
    ell_width: int
    dense_rows: torch.Tensor  # int32 [M]
    n_dense: torch.Tensor     # int32 [1]
    dense_cap: int            # routed rows the workspace holds (host value)

    def c(self) -> Hybrid:
        return Hybrid(_ptr(self.ell_val), _ptr(self.ell_col), _ptr(self.ell_nnz), int(self.ell_width),
                      _ptr(self.dense_rows), _ptr(self.n_dense), int(self.dense_cap))


def make_shape(M: int, d_model: int, d_ff: int, tile_n: int = 128, tile_cap: int = 32) -> Shape:
    return Shape(int(M), int(d_model), int(d_ff), int(tile_n), int(tile_cap))


def _pad16(n: int) -> int:
    return max(16, (n + 15) // 16 * 16)


def alloc_tiles(shape: Shape, device="cuda") -> TwellTiles:
    M, T, C = shape.M, shape.d_ff // shape.tile_n, shape.tile_cap
    # flat buffers padded to 16 bytes so every pointer handed over stays aligned
    val = torch.empty(_pad16(M * T * C * 2) // 2, dtype=torch.bfloat16, device=device)
    idx = torch.empty(_pad16(M * T * C), dtype=torch.uint8, device=device)
    cnt = torch.empty(_pad16(M * T), dtype=torch.uint8, device=device)
    nnz = torch.empty(_pad16(M * 4) // 4, dtype=torch.int32, device=device)
    return TwellTiles(val, idx, cnt, nnz)


def tiles_view(t: TwellTiles, shape: Shape):
    """(val, idx, cnt, row_nnz) reshaped to [M][T][C], [M][T][C], [M][T], [M]."""
    M, T, C = shape.M, shape.d_ff // shape.tile_n, shape.tile_cap
    return (t.val[: M * T * C].view(M, T, C), t.idx[: M * T * C].view(M, T, C),
            t.cnt[: M * T].view(M, T), t.row_nnz[:M])


def alloc_hybrid(shape: Shape, ell_width: int, device="cuda",
                 dense_cap: Optional[int] = None) -> TwellHybrid:
    """Routing buffers; dense_cap (default M, every row) is the routed-row
    capacity the workspace will be sized for."""
    M, W = shape.M, int(ell_width)
    ev = torch.empty(_pad16(M * W * 2) // 2, dtype=torch.bfloat16, device=device)
    ec = torch.empty(_pad16(M * W * 2) // 2, dtype=torch.int16, device=device)
    en = torch.empty(_pad16(M * 4) // 4, dtype=torch.int32, device=device)
    dr = torch.empty(_pad16(M * 4) // 4, dtype=torch.int32, device=device)
    nd = torch.zeros(4, dtype=torch.int32, device=device)
    return TwellHybrid(ev, ec, en, W, dr, nd, M if dense_cap is None else int(dense_cap))


def hybrid_view(h: TwellHybrid, shape: Shape):
    M, W = shape.M, h.ell_width
    return (h.ell_val[: M * W].view(M, W), h.ell_col[: M * W].view(M, W), h.ell_nnz[:M],
            h.dense_rows[:M], h.n_dense[:1])


# ------------------------------------------------------------------ entry points
def twell_pack(x, wgT, shape: Shape, out: TwellTiles, stream=None):
    t = out.c()
    _check("twell_pack", load().twell_pack(_ptr(x), _ptr(wgT), ctypes.byref(shape),
                                           ctypes.byref(t), _stream(stream)))


def twell_pack_dense(a, shape: Shape, out: TwellTiles, stream=None):
    if a.dtype == torch.float32:
        dt = 1
    elif a.dtype == torch.bfloat16:
        dt = 0
    else:
        raise ValueError("a must be float32 or bfloat16")
    t = out.c()
    _check("twell_pack_dense", load().twell_pack_dense(_ptr(a), dt, ctypes.byref(shape),
                                                       ctypes.byref(t), _stream(stream)))


def hybrid_route(tiles: TwellTiles, shape: Shape, out: TwellHybrid, stream=None):
    t, h = tiles.c(), out.c()
    _check("hybrid_route", load().hybrid_route(ctypes.byref(t), ctypes.byref(shape),
                                               ctypes.byref(h), _stream(stream)))


def twell_workspace_bytes(shape: Shape, ell_width: int, training: bool,
                          dense_cap: Optional[int] = None) -> int:
    """Workspace bytes of the sparse forward (and backward, training); room for
    dense_cap routed rows (default: every row)."""
    if dense_cap is None:
        return int(load().twell_workspace_bytes(ctypes.byref(shape), int(ell_width),
                                                int(training)))
    return int(load().twell_workspace_bytes_capped(ctypes.byref(shape), int(ell_width),
                                                   int(dense_cap), int(training)))


def twell_tiles_workspace_bytes(shape: Shape) -> int:
    return int(load().twell_tiles_workspace_bytes(ctypes.byref(shape)))


def twell_set_split_gathers(enable: bool) -> bool:
    """Split (True, the default) or fused (False) gathers for rows wider than
    1024; returns the previous setting."""
    return bool(load().twell_set_split_gathers(int(bool(enable))))


def twell_set_pair_gemm(enable: bool) -> bool:
    """CTA-pair 256 x 256 GEMM tiles (True, the default) or single-CTA
    128 x 256 tiles (False); returns the previous setting."""
    return bool(load().twell_set_pair_gemm(int(bool(enable))))


def twell_ffn_fwd(x, wgT, wuT, wd, shape: Shape, y, tiles: Optional[TwellTiles] = None,
                  route: Optional[TwellHybrid] = None, ws=None, stream=None):
    t = tiles.c() if tiles is not None else None
    h = route.c() if route is not None else None
    _check("twell_ffn_fwd", load().twell_ffn_fwd(
        _ptr(x), _ptr(wgT), _ptr(wuT), _ptr(wd), ctypes.byref(shape),
        ctypes.byref(t) if t is not None else None, ctypes.byref(h) if h is not None else None,
        _ptr(y), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def twell_ffn_fwd_noalloc(x, wgT, wuT, wd, shape: Shape, y, route: TwellHybrid, stream=None):
    """Hybrid forward whose scratch lives in the library's static device array
    (no workspace argument, nothing allocated); see include/twell.h."""
    h = route.c()
    _check("twell_ffn_fwd_noalloc", load().twell_ffn_fwd_noalloc(
        _ptr(x), _ptr(wgT), _ptr(wuT), _ptr(wd), ctypes.byref(shape), ctypes.byref(h), _ptr(y),
        _stream(stream)))


def twell_ffn_bwd(x, wgT, wuT, wd, dy, shape: Shape, route: TwellHybrid, l1_coeff: float, dx,
                  dwgT, dwuT, dwd, ws, stream=None):
    h = route.c()
    _check("twell_ffn_bwd", load().twell_ffn_bwd(
        _ptr(x), _ptr(wgT), _ptr(wuT), _ptr(wd), _ptr(dy), ctypes.byref(shape), ctypes.byref(h),
        float(l1_coeff), _ptr(dx), _ptr(dwgT), _ptr(dwuT), _ptr(dwd), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def twell_dense_workspace_bytes(shape: Shape, training: bool) -> int:
    return int(load().twell_dense_workspace_bytes(ctypes.byref(shape), int(training)))


def twell_dense_ffn_fwd(x, wgT, wuT, wd, shape: Shape, y, training: bool, ws, stream=None):
    _check("twell_dense_ffn_fwd", load().twell_dense_ffn_fwd(
        _ptr(x), _ptr(wgT), _ptr(wuT), _ptr(wd), ctypes.byref(shape), _ptr(y), int(training),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def twell_dense_ffn_bwd(x, wgT, wuT, wd, dy, shape: Shape, l1_coeff: float, dx, dwgT, dwuT, dwd,
                        ws, stream=None):
    _check("twell_dense_ffn_bwd", load().twell_dense_ffn_bwd(
        _ptr(x), _ptr(wgT), _ptr(wuT), _ptr(wd), _ptr(dy), ctypes.byref(shape), float(l1_coeff),
        _ptr(dx), _ptr(dwgT), _ptr(dwuT), _ptr(dwd), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


ACT_RELU, ACT_SILU = 0, 1


def twell_dense_ffn_fwd_act(x, wgT, wuT, wd, shape: Shape, activation: int, y, training: bool, ws,
                            stream=None):
    _check("twell_dense_ffn_fwd_act", load().twell_dense_ffn_fwd_act(
        _ptr(x), _ptr(wgT), _ptr(wuT), _ptr(wd), ctypes.byref(shape), int(activation), _ptr(y),
        int(training), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def twell_dense_ffn_bwd_act(x, wgT, wuT, wd, dy, shape: Shape, activation: int, l1_coeff: float,
                            dx, dwgT, dwuT, dwd, ws, stream=None):
    _check("twell_dense_ffn_bwd_act", load().twell_dense_ffn_bwd_act(
        _ptr(x), _ptr(wgT), _ptr(wuT), _ptr(wd), _ptr(dy), ctypes.byref(shape), int(activation),
        float(l1_coeff), _ptr(dx), _ptr(dwgT), _ptr(dwuT), _ptr(dwd), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def twell_gemm_bf16(A, B, C, M: int, N: int, K: int, a_mn_major: bool, b_mn_major: bool,
                    accumulate: bool = False, stream=None):
    c_dtype = 1 if C.dtype == torch.float32 else 0
    _check("twell_gemm_bf16", load().twell_gemm_bf16(
        _ptr(A), _ptr(B), _ptr(C), int(M), int(N), int(K), int(a_mn_major), int(b_mn_major),
        c_dtype, int(accumulate), _stream(stream)))


def twell_get_device_status(stream=None) -> int:
    out = ctypes.c_int32(0)
    _check("twell_get_device_status", load().twell_get_device_status(_stream(stream),
                                                                     ctypes.byref(out)))
    return int(out.value)


def twell_num_sms() -> int:
    return int(load().twell_num_sms())


def twell_selftest_wait_timeout(limit_us: int, stream=None):
    _check("twell_selftest_wait_timeout",
           load().twell_selftest_wait_timeout(int(limit_us), _stream(stream)))


def twell_launch_count() -> int:
    return int(load().twell_launch_count())


def twell_profile_begin(kernel: Optional[str]):
    _check("twell_profile_begin",
           load().twell_profile_begin(kernel.encode() if kernel else None))


def twell_profile_end() -> dict:
    """Stop profiling; {family: (launches, total_ms)} of the recorded launches."""
    lib = load()
    n = lib.twell_profile_end()
    if n < 0:
        raise TwellError("twell_profile_end", 5)
    out = {}
    for i in range(n):
        name, cnt, ms = ctypes.c_char_p(), ctypes.c_int32(), ctypes.c_double()
        _check("twell_profile_entry", lib.twell_profile_entry(i, ctypes.byref(name),
                                                              ctypes.byref(cnt), ctypes.byref(ms)))
        out[name.value.decode()] = (int(cnt.value), float(ms.value))
    return out
