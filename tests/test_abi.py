"""The C-ABI library loads, exports every entry point include/twell.h declares,
and rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

from activation_sparse_gated_tcgen05_gb300 import _build, twell

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "twell.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return twell.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_lists_the_boundary():
    names = declared_functions()
    for n in ("twell_pack", "twell_ffn_fwd", "twell_ffn_bwd", "hybrid_route"):
        assert n in names
    assert set(names) == set(twell.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(9):
        s = lib.twell_status_string(code)
        assert s and s != b"unknown status"
    assert lib.twell_status_string(99) == b"unknown status"


def test_host_validation_before_launch(lib):
    s = twell.make_shape(256, 256, 1024, 64, 16)
    t = twell.Tiles(16, 16, 16, 16)
    # null inputs
    assert lib.twell_pack(None, None, ctypes.byref(s), ctypes.byref(t), None) == 1
    # misaligned input
    assert lib.twell_pack(8, 16, ctypes.byref(s), ctypes.byref(t), None) == 3
    # unsupported shapes
    for bad in (twell.make_shape(256, 100, 1024, 64, 16), twell.make_shape(256, 256, 1000, 64, 16),
                twell.make_shape(256, 256, 1024, 32, 16), twell.make_shape(256, 256, 1024, 64, 0),
                twell.make_shape(256, 256, 1024, 64, 65)):
        assert lib.twell_pack(16, 16, ctypes.byref(bad), ctypes.byref(t), None) == 2
    assert lib.twell_pack(16, 16, ctypes.byref(twell.make_shape(-1, 256, 1024, 64, 16)),
                          ctypes.byref(t), None) == 1
    # exactly one of tiles / route
    assert lib.twell_ffn_fwd(16, 16, 16, 16, ctypes.byref(s), None, None, 16, None, 0, None) == 1
    # workspace too small
    h = twell.Hybrid(16, 16, 16, 8, 16, 16, 256)
    assert lib.twell_ffn_fwd(16, 16, 16, 16, ctypes.byref(s), None, ctypes.byref(h), 16, 16, 8,
                             None) == 7
    # a negative routed-row capacity
    hneg = twell.Hybrid(16, 16, 16, 8, 16, 16, -1)
    assert lib.hybrid_route(ctypes.byref(t), ctypes.byref(s), ctypes.byref(hneg), None) == 1
    assert lib.twell_ffn_fwd(16, 16, 16, 16, ctypes.byref(s), None, ctypes.byref(hneg), 16, 16,
                             1 << 30, None) == 1
    # TwELL forward of wide rows: a workspace that is given must hold h
    wide = twell.make_shape(256, 2048, 1024, 64, 16)
    assert lib.twell_ffn_fwd(16, 16, 16, 16, ctypes.byref(wide), ctypes.byref(t), None, 16, 16,
                             8, None) == 7
    assert lib.twell_pack_dense(16, 3, ctypes.byref(s), ctypes.byref(t), None) == 1
    assert lib.twell_gemm_bf16(16, 16, 16, 10, 12, 16, 0, 0, 0, 0, None) == 2
    # dense comparator: unknown activation; SiLU has no L1 term
    assert lib.twell_dense_ffn_fwd_act(16, 16, 16, 16, ctypes.byref(s), 2, 16, 1, 16, 1 << 30,
                                       None) == 1
    assert lib.twell_dense_ffn_bwd_act(16, 16, 16, 16, 16, ctypes.byref(s), 1, 2e-5, 16, 16, 16,
                                       16, 16, 1 << 30, None) == 1
    assert lib.twell_dense_ffn_bwd_act(16, 16, 16, 16, 16, ctypes.byref(s), 1, 0.0, 16, 16, 16,
                                       16, 16, 8, None) == 7


def test_pair_gemm_switch(lib):
    assert twell.twell_set_pair_gemm(False) is True   # the default is on
    assert twell.twell_set_pair_gemm(True) is False
    assert twell.twell_set_pair_gemm(True) is True


def test_split_gathers_switch(lib):
    assert twell.twell_set_split_gathers(False) is True   # the default is on
    assert twell.twell_set_split_gathers(True) is False
    assert twell.twell_set_split_gathers(True) is True


def test_workspace_sizes(lib):
    s = twell.make_shape(16384, 1024, 4096, 128, 32)
    inf = twell.twell_workspace_bytes(s, 30, False)
    tr = twell.twell_workspace_bytes(s, 30, True)
    assert 0 < inf < tr
    assert twell.twell_workspace_bytes(twell.make_shape(16, 100, 1024, 64, 16), 4, True) == 0
    # the dense-backup buffers scale with the routed-row capacity
    assert twell.twell_workspace_bytes(s, 30, True, dense_cap=16384) == tr
    assert twell.twell_workspace_bytes(s, 30, True, dense_cap=1 << 20) == tr
    c512 = twell.twell_workspace_bytes(s, 30, True, dense_cap=512)
    c0 = twell.twell_workspace_bytes(s, 30, True, dense_cap=0)
    assert 0 < c0 < c512 < tr / 2
    assert twell.twell_workspace_bytes(s, 30, True, dense_cap=-1) == 0
    # 512 routed rows (4 tiles) of x, dY, h hi+lo, g, u fp32, du/da hi+lo
    f, d = 4096, 1024
    assert c512 - c0 >= 512 * (2 * d * 2 + 2 * f * 2 + f * 2 + f * 4 + 4 * f * 2)
    assert twell.twell_dense_workspace_bytes(s, True) >= 5 * 16384 * 4096 * 2
    # TwELL forward: no workspace up to d_model = 1024, then h per slot + the y carry
    assert twell.twell_tiles_workspace_bytes(s) == 0
    wide = twell.make_shape(32768, 2048, 8192, 128, 32)
    assert twell.twell_tiles_workspace_bytes(wide) >= 4 * 32768 * (64 * 32 + 2048)
    assert twell.twell_tiles_workspace_bytes(twell.make_shape(16, 100, 1024, 64, 16)) == 0


def test_gather_probe_lives_in_its_own_library(lib):
    """The benchmark's row-gather probe is a separate library, not part of
    the FFN library's ABI."""
    assert not hasattr(lib, "twell_probe_gather")
    from activation_sparse_gated_tcgen05_gb300 import probe

    plib = probe.load()
    assert hasattr(plib, "twell_probe_gather")
    # host-side checks: null table, output shorter than one word per warp
    assert plib.twell_probe_gather(None, 4, 16, 16, 1, 16, 8, 1, None) == 1
    assert plib.twell_probe_gather(16, 4, 16, 16, 1, 16, 7, 1, None) == 1
    assert plib.twell_probe_gather(16, 4, 24, 16, 1, 16, 8, 1, None) == 2
    assert plib.twell_probe_gather(8, 4, 16, 16, 1, 16, 8, 1, None) == 3
