"""CPU-only: the C-ABI library builds, loads, exports every declared symbol,
and its host-side logic (argument checks, path choice, rasteriser, workspace
sizing) behaves as documented.  Nothing here launches a kernel."""
import os
import re

import pytest

import tiled_tensor_core_03_gb300 as gr
from tiled_tensor_core_03_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if _build.needs_build():
        _build.build()
    return gr.lib()


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_entry_points():
    names = declared_functions()
    for want in ("gemm_relu_f16", "gemm_relu_f16_splitk", "gemm_relu_f16_splitk_workspace_bytes",
                 "gemm_relu_status", "gemm_relu_strerror"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_strerror(lib):
    for code in range(7):
        assert gr.strerror(code)
    assert gr.strerror(999) == "unknown status"


def test_streamk_hook_arguments(lib):
    assert gr.gemm_relu_debug_streamk(4) == gr.ERR_INVALID_ARG
    assert gr.gemm_relu_debug_streamk(-1) == gr.ERR_INVALID_ARG
    for mode in (gr.SK_HEAD_LATE, gr.SK_TAIL_LATE, gr.SK_HEAD_PUBLISHES, gr.SK_NORMAL):
        assert gr.gemm_relu_debug_streamk(mode) == gr.OK
    for bad in (1, 9, -1):
        assert gr.gemm_relu_debug_streamk_pieces(bad) == gr.ERR_INVALID_ARG
    for ok in (8, 3, 2, 0):
        assert gr.gemm_relu_debug_streamk_pieces(ok) == gr.OK


def test_panel_hook_arguments(lib):
    assert gr.gemm_relu_debug_set_panel(-128) == gr.ERR_INVALID_ARG
    assert gr.gemm_relu_debug_set_panel(200) == gr.ERR_INVALID_ARG
    assert gr.gemm_relu_debug_set_panel(384) == gr.OK
    assert gr.gemm_relu_debug_set_panel(0) == gr.OK


def test_invalid_arguments_rejected_on_host(lib):
    c = 0x1000
    assert gr.gemm_relu_f16(c, c, c, -1, 4, 4) == gr.ERR_INVALID_ARG
    assert gr.gemm_relu_f16(c, c, c, 4, 4, 1 << 31) == gr.ERR_INVALID_ARG
    assert gr.gemm_relu_f16(c, c, None, 4, 4, 4) == gr.ERR_INVALID_ARG
    assert gr.gemm_relu_f16(None, c, c, 4, 4, 4) == gr.ERR_INVALID_ARG
    assert gr.gemm_relu_f16(c + 1, c, c, 4, 4, 4) == gr.ERR_INVALID_ARG   # odd address
    assert gr.gemm_relu_f16_splitk(c, c, c, 4, 4, 4, 0, c, 1 << 20) == gr.ERR_WORKSPACE
    # empty outputs need no device and no pointers
    assert gr.gemm_relu_f16(None, None, None, 0, 5, 5) == gr.OK
    assert gr.gemm_relu_f16(None, None, None, 5, 0, 5) == gr.OK


def test_path_choice(lib):
    a = 0x10000
    assert gr.gemm_relu_f16_path(a, a, a, 128, 256, 64) == gr.PATH_TMA
    assert gr.gemm_relu_f16_path(a, a, a, 1537, 1023, 777) == gr.PATH_LSU   # pitches not 16 B
    assert gr.gemm_relu_f16_path(a + 8, a, a, 128, 256, 64) == gr.PATH_LSU  # A not 16-B aligned
    assert gr.gemm_relu_f16_path(a, a, a, 128, 256, 60) == gr.PATH_LSU      # K*2 % 16 != 0
    assert gr.gemm_relu_f16_path(a, a, a, 128, 250, 64) == gr.PATH_LSU
    assert gr.gemm_relu_f16_path(a, a, a, 0, 256, 64) == gr.PATH_NONE
    assert gr.gemm_relu_f16_path(a, a, a, 8, 8, 0) == gr.PATH_NONE
    assert gr.gemm_relu_f16_path(a, a, a, -8, 8, 8) == -1


@pytest.mark.parametrize("m_tiles,n_tiles,panel", [(32, 16, 8), (13, 4, 8), (1, 1, 8), (7, 3, 4),
                                                   (9, 5, 1), (3, 11, 16), (33, 2, 4)])
def test_rasteriser_is_a_bijection(lib, m_tiles, n_tiles, panel):
    seen = set()
    for t in range(m_tiles * n_tiles):
        mb, nb = gr.gemm_relu_tile_coord(t, m_tiles, n_tiles, panel)
        assert 0 <= mb < m_tiles and 0 <= nb < n_tiles
        seen.add((mb, nb))
    assert len(seen) == m_tiles * n_tiles
    with pytest.raises(ValueError):
        gr.gemm_relu_tile_coord(m_tiles * n_tiles, m_tiles, n_tiles, panel)


def test_rasteriser_panel_order(lib):
    # panel 4, column order: ids 0..3 walk down M in N block 0, 4..7 in N block 1
    coords = [gr.gemm_relu_tile_coord(t, 8, 3, 4) for t in range(12)]
    assert coords[:5] == [(0, 0), (1, 0), (2, 0), (3, 0), (0, 1)]
    assert coords[11] == (3, 2)
    assert gr.gemm_relu_tile_coord(12, 8, 3, 4) == (4, 0)      # second panel


def test_splitk_workspace_size(lib):
    # split 2, 4 or 8 after clamping: reduced inside a cluster, no workspace
    assert gr.gemm_relu_f16_splitk_workspace_bytes(16, 8192, 8192, 8) == 0
    assert gr.gemm_relu_f16_splitk_workspace_bytes(16, 8192, 8192, 4) == 0
    assert gr.gemm_relu_f16_splitk_workspace_bytes(64, 128, 600, 4) == 0
    assert gr.gemm_relu_f16_splitk_workspace_bytes(16, 128, 8192, 32) == 0
    # M > 64, odd splits, or splits * R > 512: two-stage, split_k * M * N fp32
    assert gr.gemm_relu_f16_splitk_workspace_bytes(200, 128, 600, 2) == 2 * 200 * 128 * 4
    assert gr.gemm_relu_f16_splitk_workspace_bytes(64, 128, 8192, 16) == 16 * 64 * 128 * 4
    # other splits: split_k * M * N fp32 partials
    assert gr.gemm_relu_f16_splitk_workspace_bytes(16, 8192, 8192, 3) == 3 * 16 * 8192 * 4
    assert gr.gemm_relu_f16_splitk_workspace_bytes(16, 8192, 8192, 1) == 0
    # M <= 32 works in 256-wide k stages: K = 600 has 3, so split 8 clamps to 3
    assert gr.gemm_relu_f16_splitk_workspace_bytes(16, 128, 600, 8) == 3 * 16 * 128 * 4
    assert gr.gemm_relu_f16_splitk_workspace_bytes(16, 128, 100, 8) == 0     # one stage
    # 32 < M <= 64 works in 128-wide stages, larger M in 64-wide ones
    assert gr.gemm_relu_f16_splitk_workspace_bytes(64, 128, 600, 8) == 5 * 64 * 128 * 4
    assert gr.gemm_relu_f16_splitk_workspace_bytes(200, 128, 600, 16) == 10 * 200 * 128 * 4
    # the two-stage form, when forced, always takes a workspace
    assert gr.gemm_relu_debug_force_split(gr.SPLIT_TWO_STAGE) == gr.OK
    try:
        assert gr.gemm_relu_f16_splitk_workspace_bytes(16, 8192, 8192, 8) == 8 * 16 * 8192 * 4
        assert gr.gemm_relu_f16_splitk_workspace_bytes(64, 128, 600, 4) == 4 * 64 * 128 * 4
    finally:
        assert gr.gemm_relu_debug_force_split(gr.SPLIT_AUTO) == gr.OK
    assert gr.gemm_relu_debug_force_split(2) == gr.ERR_INVALID_ARG
    assert gr.gemm_relu_f16_splitk_workspace_bytes(0, 8, 8, 2) == 0
    assert gr.gemm_relu_f16_splitk_workspace_bytes(8, 8, 8, 0) == 0


def test_streamk_plan_rules(lib):
    """The stream-K schedule chosen per shape on a 152-SM GPU (host-only):
    multi-wave schedules only where the idle part of the last wave,
    (ceil(W) - W) x k blocks, reaches 40; sub-wave schedules for M > 64 with
    pieces = k blocks / 128 + 1 (at least 2) per tile, pieces x tiles <= SMs,
    at least 32 k blocks saved and a shared operand under 64 MB; nothing on
    rows TMA cannot describe (those are staged and planned as TMA rows)."""
    plan = gr.streamk_plan
    # CTA pairs, multi-wave: 4096^3 (W = 3.37 on 76 pairs) keeps it; 2304^2
    # and 2560^2 at K = 4096 (W = 1.07, 1.32) too; short K or a nearly full
    # last wave declines
    assert plan(4096, 4096, 4096, 152) == (152, 152, True)
    assert plan(2304, 2304, 4096, 152) == (0, 152, True)
    assert plan(2560, 2560, 4096, 152) == (0, 152, True)
    for shape in [(3072, 3072, 3072), (2304, 2304, 1024), (4096, 4096, 2048), (4608, 4608, 2048)]:
        assert plan(*shape, 152)[0] == -1, shape
    # single CTAs, sub-wave: 2 / 3 / 5 pieces a tile on pieces x tiles CTAs
    assert plan(200, 3000, 4096, 152) == (0, 96, False)
    assert plan(128, 2048, 16384, 152) == (0, 48, False)
    assert plan(100, 1024, 32768, 152) == (0, 40, False)
    # declined: too few k blocks saved; a 105 MB B shared by two rows of
    # tiles; more than 152 CTAs; skinny rows (split-K / GEMV); unaligned rows
    for shape in [(1024, 1024, 1024), (192, 6400, 8192), (128, 12800, 8192), (16, 8192, 8192)]:
        assert plan(*shape, 152)[0] == -1, shape
    assert plan(1537, 1023, 777, 152, path=gr.PATH_LSU)[0] == -1
    assert plan(200, 3000, 4096, 152, path=gr.PATH_LSU)[0] == -1
    # the SM count decides: half the SMs leave no room for two pieces of 96 tiles
    assert plan(200, 3000, 4096, 76)[0] == -1
    try:
        assert gr.gemm_relu_debug_streamk_pieces(4) == gr.OK
        assert plan(128, 4096, 8192, 152) == (0, 128, False)
        assert gr.gemm_relu_debug_force_kernel(gr.FORCE_ONE_CTA_256) == gr.OK
        assert plan(2304, 2304, 4096, 152) == (0, 152, False)    # 162 tiles of 128 x 256
    finally:
        gr.gemm_relu_debug_streamk_pieces(0)
        gr.gemm_relu_debug_force_kernel(gr.FORCE_AUTO)
    for bad in [(0, 64, 64, 152), (64, 64, 64, 1)]:
        with pytest.raises(ValueError):
            plan(*bad)
    with pytest.raises(ValueError):
        plan(64, 64, 64, 152, path=3)
