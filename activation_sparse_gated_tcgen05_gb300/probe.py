"""ctypes binding of libtwell_probe.so, the benchmark's row-gather bandwidth
probe (warps read whole rows of a table at given ids with 16-byte loads, the
access pattern of the sparse gather kernels).  A measurement helper: it is
not part of the FFN library or its C ABI."""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

_lib = None


def load():
    global _lib
    if _lib is None:
        if not os.path.exists(_build.PROBE_LIB):
            raise RuntimeError("libtwell_probe.so not found: run __graft_entry__.build()")
        lib = ctypes.CDLL(_build.PROBE_LIB)
        P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.twell_probe_gather.restype = I32
        lib.twell_probe_gather.argtypes = [P, I64, I32, P, I64, P, I64, I32, P]
        _lib = lib
    return _lib


def gather(table: torch.Tensor, row_bytes: int, idx: torch.Tensor, out: torch.Tensor,
           blocks: int, stream=None) -> None:
    """Gather rows idx (int32) of `table` (row_bytes each); `out` (int32 or
    uint32, at least blocks * 8 words) receives one folded word per warp."""
    for t in (table, idx, out):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous and on the GPU")
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream.cuda_stream
    rows = table.numel() * table.element_size() // int(row_bytes)
    st = load().twell_probe_gather(table.data_ptr(), rows, int(row_bytes), idx.data_ptr(),
                                   idx.numel(), out.data_ptr(),
                                   out.numel() * out.element_size() // 4, int(blocks), s)
    if st != 0:
        raise RuntimeError("twell_probe_gather failed with status %d" % st)
