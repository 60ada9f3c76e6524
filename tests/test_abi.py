"""The C ABI without a GPU: the library loads, exports every function the header
declares, and rejects bad arguments before touching the device.  Also the host-side
work decomposition (pieces of units per CTA)."""
import ctypes
import os
import subprocess

import pytest

from bit_weight_streaming_q4_gb300 import build as qbuild
from bit_weight_streaming_q4_gb300 import qmm as Q


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return Q.load()


def test_header_declares_expected_api():
    names = Q.header_functions()
    assert names == sorted(["qmm_default_options", "qmm_create", "qmm_run", "qmm_run_host",
                            "qmm_get_error", "qmm_get_info", "qmm_destroy", "qmm_status_str",
                            "qmm_step_create", "qmm_step_launch", "qmm_step_launch_host", "qmm_step_destroy",
                            "qmm_run_noalloc", "qmm_run_argmax", "qmm_attn_workspace_bytes",
                            "qmm_attn_decode"])


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", Q.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in Q.header_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings(lib):
    for code in range(10):
        s = lib.qmm_status_str(code)
        assert s and s != b"unknown status"
    assert lib.qmm_status_str(99) == b"unknown status"


def test_default_options(lib):
    o = Q.Options()
    lib.qmm_default_options(ctypes.byref(o))
    assert (o.m_max, o.backend, o.ctas_per_sm, o.host_io, o.format, o.wait_limit_us) == (16, 0, 0, 0, 0, 0)


def test_argument_errors_need_no_device(lib):
    h = ctypes.c_void_p()
    buf = (ctypes.c_uint8 * 144)()
    o = Q.default_options()
    assert lib.qmm_create(None, buf, 1, 256, 0, ctypes.byref(o), None) == 1
    assert lib.qmm_create(ctypes.byref(h), None, 1, 256, 0, ctypes.byref(o), None) == 1
    assert lib.qmm_create(ctypes.byref(h), buf, 1, 300, 0, ctypes.byref(o), None) == 2
    assert lib.qmm_create(ctypes.byref(h), buf, 0, 256, 0, ctypes.byref(o), None) == 2
    assert lib.qmm_create(ctypes.byref(h), buf, 1, -256, 0, ctypes.byref(o), None) == 2
    bad = Q.default_options(m_max=0)
    assert lib.qmm_create(ctypes.byref(h), buf, 1, 256, 0, ctypes.byref(bad), None) == 1
    # an unknown block format, and a Q6_K / Q8_0 handle on the mma.sync backend
    for fmt, be in ((3, 0), (-1, 0), (1, 1), (2, 1)):
        o2 = Q.default_options(backend=be, format=fmt)
        assert lib.qmm_create(ctypes.byref(h), buf, 1, 256, 0, ctypes.byref(o2), None) == 1
    misaligned = ctypes.addressof(buf) | 1
    assert lib.qmm_create(ctypes.byref(h), misaligned, 1, 256, 1, ctypes.byref(o), None) == 3
    # no handle exists: every handle call reports BAD_HANDLE
    assert lib.qmm_run(None, buf, 1, buf, None) == 7
    assert lib.qmm_run(ctypes.c_void_p(0x1000), buf, 1, buf, None) == 7
    assert lib.qmm_destroy(ctypes.c_void_p(0x1000)) == 7
    assert lib.qmm_get_error(None) == 7
    assert lib.qmm_step_launch(None, None) == 7
    assert lib.qmm_step_launch_host(None, buf, buf, None, None, None) == 7
    assert lib.qmm_step_launch_host(ctypes.c_void_p(0x1000), buf, buf, None, None, None) == 7
    assert lib.qmm_run_argmax(None, buf, 1, buf, buf, None) == 7
    assert lib.qmm_run_argmax(ctypes.c_void_p(0x1000), buf, 1, buf, buf, None) == 7
    assert lib.qmm_step_destroy(None) == 7


def test_no_device_is_reported(lib):
    """Without an sm_103 GPU qmm_create reports NO_DEVICE instead of crashing."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    buf = (ctypes.c_uint8 * 144)()
    o = Q.default_options()
    assert lib.qmm_create(ctypes.byref(h), buf, 1, 256, 0, ctypes.byref(o), None) == 8


def _piece_of(u, units, grid):
    return ((u + 1) * grid + units - 1) // units - 1


@pytest.mark.parametrize("units,grid", [(10, 3), (2048, 152), (1920, 152), (189920, 152),
                                        (7, 7), (152, 152), (3, 1), (1000003, 304)])
def test_pieces_partition_units(units, grid):
    bounds = [c * units // grid for c in range(grid + 1)]
    assert bounds[0] == 0 and bounds[-1] == units
    sizes = [b - a for a, b in zip(bounds, bounds[1:])]
    assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1
    probe = sorted({0, units - 1, units // 2, *bounds[1:-1], *(b - 1 for b in bounds[1:-1])})
    for u in probe:
        c = _piece_of(u, units, grid)
        assert bounds[c] <= u < bounds[c + 1], (u, c)


@pytest.mark.parametrize("mats,grid", [([(40, 20)], 152), ([(40, 68)], 152), ([(1187, 20)], 152),
                                       ([(64, 20), (40, 24), (272, 20), (40, 68)] * 3 + [(1187, 20)], 152),
                                       ([(2, 1), (1, 3), (5, 2)], 4), ([(3, 256)], 7)])
def test_split_tile_bookkeeping(mats, grid):
    """Both kernels' split-K bookkeeping, restated on the host: a launch of matrices (tiles, kb)
    cut into `grid` pieces.  A tile shared by pieces pa..pb is reduced by pa; each other piece
    writes one partial into its CTA's writer slot.  That slot suffices because a piece can
    share, without reducing, only its first tile.  The reducer pa reaches the tile at the end
    of its piece (the tile is pa's last tile), so each piece is pa for at most one shared tile
    and one more slot holds a partial that pa parks when it must leave the sum to the last
    CTA to arrive (tcgen05 kernel)."""
    units = sum(t * kb for t, kb in mats)
    grid = min(grid, units)
    start = [c * units // grid for c in range(grid + 1)]
    partials, parked = {}, {}
    base = 0
    for tiles, kb in mats:
        for tile in range(tiles):
            t0, t1 = base + tile * kb, base + (tile + 1) * kb
            pa, pb = _piece_of(t0, units, grid), _piece_of(t1 - 1, units, grid)
            if pa == pb:
                continue
            # the reducer's piece ends inside the tile: it is pa's last tile
            assert t0 < start[pa + 1] <= t1
            assert pa not in parked, (pa, parked[pa], (base, tile))
            parked[pa] = (base, tile)
            for c in range(pa + 1, pb + 1):
                # each writer starts inside the tile: it is that piece's first tile
                assert t0 < start[c] < t1
                assert c not in partials, (c, partials[c], (base, tile))
                partials[c] = (base, tile)
        base += tiles * kb


def test_library_not_built_raises(tmp_path):
    saved = Q._lib
    try:
        Q._lib = None
        with pytest.raises(RuntimeError, match="not built"):
            Q.load(str(tmp_path / "missing.so"))
    finally:
        Q._lib = saved


def test_attention_arguments_without_device(lib):
    """The attention entry's workspace size (fixed by the dimensions and the row count) and
    the argument errors it reports before any launch."""
    dims = Q.AttnDims(48, 8, 4, 400, 1600)
    nbytes = ctypes.c_int64()
    # agents x KV heads x runs x query tiles x 24 queries x (128 + 4) floats.  Runs are planned
    # for at most 1024 resident CTAs: at most 1024 // 32 = 32 runs, so runs of
    # ceil(400 / 32) = 13 pages, of which 400 pages make 31.  Query tiles: all rows in one agent,
    # 6 queries per row and KV head, 24 per tile.
    for rows, tiles in ((1, 1), (4, 1), (5, 2), (8, 2), (12, 3), (64, 16)):
        assert lib.qmm_attn_workspace_bytes(ctypes.byref(dims), rows, ctypes.byref(nbytes)) == 0
        assert nbytes.value == 4 * 8 * 31 * tiles * 24 * 132 * 4, rows
    wide = Q.AttnDims(48, 8, 128, 20, 1600)  # 1024 (agent, KV head) pairs: one run each
    assert lib.qmm_attn_workspace_bytes(ctypes.byref(wide), 3, ctypes.byref(nbytes)) == 0
    assert nbytes.value == 128 * 8 * 1 * 1 * 24 * 132 * 4
    short = Q.AttnDims(48, 8, 1, 5, 1600)  # at most one run per page
    assert lib.qmm_attn_workspace_bytes(ctypes.byref(short), 3, ctypes.byref(nbytes)) == 0
    assert nbytes.value == 1 * 8 * 5 * 1 * 24 * 132 * 4
    for bad in (Q.AttnDims(48, 7, 4, 400, 1600), Q.AttnDims(0, 8, 4, 400, 1600), Q.AttnDims(48, 8, 0, 400, 1600),
                Q.AttnDims(48, 8, 4, 0, 1600), Q.AttnDims(48, 8, 4, 400, 0)):
        assert lib.qmm_attn_workspace_bytes(ctypes.byref(bad), 3, ctypes.byref(nbytes)) == 1
    for rows in (0, -1, (1 << 24) + 1):
        assert lib.qmm_attn_workspace_bytes(ctypes.byref(dims), rows, ctypes.byref(nbytes)) == 1
    # a bound on any agent's rows sizes the query tiles: 12 rows, at most 3 per agent -> 1 tile
    hinted = Q.AttnDims(48, 8, 4, 400, 1600, 3)
    assert lib.qmm_attn_workspace_bytes(ctypes.byref(hinted), 12, ctypes.byref(nbytes)) == 0
    assert nbytes.value == 4 * 8 * 31 * 1 * 24 * 132 * 4
    hinted = Q.AttnDims(48, 8, 4, 400, 1600, 50)  # a bound above the rows changes nothing
    assert lib.qmm_attn_workspace_bytes(ctypes.byref(hinted), 12, ctypes.byref(nbytes)) == 0
    assert nbytes.value == 4 * 8 * 31 * 3 * 24 * 132 * 4
    for bad in (Q.AttnDims(48, 8, 4, 400, 1600, -1), Q.AttnDims(48, 8, 4, 400, 1600, 0, 1)):
        assert lib.qmm_attn_workspace_bytes(ctypes.byref(bad), 12, ctypes.byref(nbytes)) == 1
    buf = (ctypes.c_uint8 * 64)()
    assert lib.qmm_attn_decode(ctypes.byref(dims), None, buf, buf, buf, buf, 1, buf, buf, 10**9, buf, None) == 1
    assert lib.qmm_attn_decode(ctypes.byref(dims), buf, buf, buf, buf, buf, 0, buf, buf, 10**9, buf, None) == 1
    assert lib.qmm_attn_decode(ctypes.byref(dims), buf, buf, buf, buf, buf, 1, buf, buf, 16, buf, None) in (3, 9)
