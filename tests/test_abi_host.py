"""Host-side tests of the C ABI: no kernel is launched and no GPU is needed.

The library must load, export every entry point include/convgb.h declares,
derive shapes, sizes and paths exactly as the oracle and the pages say, and
reject bad arguments before touching the GPU.
"""
import ctypes
import os
import re

import pytest

import oracle
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import indirect_implicit_gemm_gb300 as g
    return g


def header_symbols():
    text = open(os.path.join(ROOT, "include", "convgb.h")).read()
    return sorted(set(re.findall(r"^CONVGB_API [^(]*?\b([a-z_0-9]+)\(", text, re.M)))


def test_library_exports_every_declared_symbol(lib):
    declared = header_symbols()
    assert len(declared) >= 16
    assert sorted(lib.EXPORTED_SYMBOLS) == declared
    so = ctypes.CDLL(lib.library_path)
    for name in declared:
        assert hasattr(so, name), name


def test_library_has_no_libcuda_link_dependency(lib):
    """The driver API is reached at run time; loading needs no libcuda.so here."""
    import subprocess
    out = subprocess.run(["readelf", "-d", lib.library_path], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out


def test_status_strings(lib):
    so = lib.load()
    for s in range(7):
        assert so.convgb_status_string(s)
    assert so.convgb_status_string(99) == b"unknown status"
    assert so.convgb_version() >= 100


SHAPES = [(56, 3, 1, 1, 1), (224, 7, 2, 3, 1), (224, 11, 4, 2, 1), (28, 3, 1, 2, 2), (7, 7, 1, 0, 1),
          (27, 5, 1, 2, 1), (56, 1, 2, 0, 1), (150, 3, 1, 1, 1), (5, 3, 1, 0, 2), (10, 4, 3, 1, 2),
          (1, 1, 1, 0, 1), (9, 2, 5, 0, 3), (13, 6, 3, 4, 2)]


@pytest.mark.parametrize("L,K,s,p,d", SHAPES)
def test_output_dims_match_oracle(lib, L, K, s, p, d):
    ho, wo = lib.output_dims(L, L + 1, K, K, s, p, d)
    assert ho == oracle.output_size(L, K, s, p, d)
    assert wo == oracle.output_size(L + 1, K, s, p, d)


def test_output_dims_reject_empty(lib):
    with pytest.raises(lib.ConvgbError):
        lib.output_dims(3, 3, 5, 5, 1, 0, 1)
    with pytest.raises(lib.ConvgbError):
        lib.output_dims(8, 8, 3, 3, 0, 1, 1)


@pytest.mark.parametrize("cfg", workloads.ALL, ids=lambda c: c.name)
def test_sizes_and_workspace_below_im2col(lib, cfg):
    a = (cfg.N, cfg.C_in, cfg.H, cfg.W)
    geo = (cfg.KH, cfg.KW, cfg.stride, cfg.pad, cfg.dilation)
    im2col = lib.im2col_bytes(*a, *geo)
    assert im2col == 2 * oracle.im2col_elements(*a, *geo)
    assert lib.im2win_bytes(*a, *geo) == 2 * oracle.im2win_elements(*a, *geo)
    ho, wo = oracle.output_size(cfg.H, cfg.KH, cfg.stride, cfg.pad, cfg.dilation), \
        oracle.output_size(cfg.W, cfg.KW, cfg.stride, cfg.pad, cfg.dilation)
    assert lib.indirection_buffer_bytes(cfg.H, cfg.W, *geo) == ho * wo * cfg.KH * cfg.KW * 4
    ws = lib.workspace_size(cfg.N, cfg.C_in, cfg.H, cfg.W, cfg.C_out, *geo)
    assert ws < im2col, (ws, im2col)


def expected_path(c):
    if c.KH == 1 or "fullspatial" in c.name:
        return 2  # dense GEMM
    if c.C_in % 8:
        Ho = oracle.output_size(c.H, c.KH, c.stride, c.pad, c.dilation)
        Wo = oracle.output_size(c.W, c.KW, c.stride, c.pad, c.dilation)
        # staged window in shared memory: C_in <= 4, stride 1/2/4, undilated, one
        # output row's K blocks within a 128-row tile, rows and weights in whole
        # 16-byte copies, one column tile
        nkb = -(-c.KW // c.stride)
        steps = (nkb - 1) * 4 + -(-((c.KW - c.stride * (nkb - 1)) * (64 // c.stride)) // 16) \
            if c.stride in (1, 2, 4) else 99
        if (c.C_in == 3 and c.stride in (1, 2, 4) and c.dilation == 1 and steps <= 16 and
                Wo + nkb - 1 <= 128 and (c.W * c.C_in * 2) % 16 == 0 and
                (c.C_out * c.KH * c.KW * c.C_in * 2) % 16 == 0 and c.C_out <= 256):
            return 7
        # window-order (im2win) buffer while it stays under half of im2col, else stem
        KC = (c.KH * c.C_in + 7) // 8 * 8
        W_used = (Wo - 1) * c.stride + (c.KW - 1) * c.dilation + 1
        buf = c.N * Ho * W_used * KC * 2
        im2col = c.N * Ho * Wo * c.KH * c.KW * c.C_in * 2
        if (c.C_in < 16 and c.dilation == 1 and Wo <= 128 and
                W_used * KC * 2 + c.KH * c.W * c.C_in * 2 + 16 <= 48 * 1024 and
                buf < im2col // 2):
            return 6  # im2win
        return 3  # stem
    wv = oracle.output_size(c.W, c.KW, c.stride, c.pad, c.dilation) + (c.KW - 1) * c.dilation
    if c.stride == 1 and c.C_in % 64 == 0 and wv <= 128 and (c.KW - 1) * c.dilation <= 8:
        return 4  # window
    # taps folded into the MMA's columns: 32 input channels, segments of
    # G = 32 - (KW-1)d output pixels, at least 12 of them per segment on average
    G = 32 - (c.KW - 1) * c.dilation
    Wo = oracle.output_size(c.W, c.KW, c.stride, c.pad, c.dilation)
    if (c.stride == 1 and c.C_in == 32 and c.C_out % 32 == 0 and c.KW <= 5 and c.KH <= 7 and
            G >= 8 and c.KW * c.C_out <= 256 and c.W >= 32 and c.dilation <= 8 and
            Wo >= 12 * -(-Wo // G)):
        return 8
    return 1  # indirection-buffer gather


@pytest.mark.parametrize("cfg,path", [
    (workloads.TINY, 3), (workloads.RESNET_3X3, 4), (workloads.POINTWISE_S1, 2),
    (workloads.POINTWISE_S2, 2), (workloads.STEM_7X7, 7), (workloads.STRIDED_3X3, 1),
] + [(c, expected_path(c)) for c in workloads.SWEEP], ids=lambda v: getattr(v, "name", str(v)))
def test_path_selection(lib, cfg, path):
    got = lib.select_path(cfg.N, cfg.C_in, cfg.H, cfg.W, cfg.C_out, cfg.KH, cfg.KW, cfg.stride,
                          cfg.pad, cfg.dilation)
    assert got == path


def test_winfold_selection_and_plan(lib):
    # 32 -> 32 3x3 at 150x150: segments of 30 output pixels, five per output row
    pl = lib.plan_info(128, 32, 150, 150, 32, 3, 3, 1, 1, 1)
    assert (pl["path"], pl["a_mode"], pl["segment_outputs"], pl["tile_rows"]) == (8, 17, 30, 0)
    # 5x5: the instantiation with tap loops for up to 7 x 5
    assert lib.plan_info(128, 32, 150, 150, 32, 5, 5, 1, 2, 1)["a_mode"] == 16
    # 8-row units (3x3, 96-column MMA) x segments
    assert pl["segment_rows"] == 8
    assert pl["m_tiles"] == 128 * 19 * 5 and pl["k_blocks"] == 1
    assert pl["weights_resident"] == 1 and pl["splits"] == 1 and pl["tma_store"] == 0
    assert lib.workspace_size(128, 32, 150, 150, 32, 3, 3, 1, 1, 1) == 0
    # rows narrower than a 32-pixel segment stay on the gather path
    assert lib.select_path(4, 32, 8, 8, 32, 3, 3, 1, 1, 1) == 1
    assert lib.select_path(4, 32, 31, 31, 32, 3, 3, 1, 1, 1) == 1
    assert lib.select_path(4, 32, 32, 32, 32, 3, 3, 1, 1, 1) == 8
    # C_out not a multiple of 32, stride 2, or KW*C_out past 256: not folded
    assert lib.select_path(4, 32, 40, 40, 48, 3, 3, 1, 1, 1) == 1
    assert lib.select_path(4, 32, 40, 40, 32, 3, 3, 2, 1, 1) == 1
    assert lib.select_path(4, 32, 40, 40, 128, 3, 3, 1, 1, 1) == 1
    with pytest.raises(lib.ConvgbError):
        lib.plan_info(4, 32, 40, 40, 128, 3, 3, 1, 1, 1, path=lib.PATH_WINFOLD)


def test_window_plans_ring_depth(lib):
    # A window A slot holds only the staged rows (two boxes of 58 pixels on the
    # 64 -> 128 3x3 layer at 56x56) rather than every row the MMAs read, so a
    # fourth slot fits beside the 144 KB of resident weights; the fixed-plan
    # kernel (resident weights, TMA-store epilogue in 64-column chunks) runs it.
    pl = lib.plan_info(32, 64, 56, 56, 128, 3, 3, 1, 1, 1)
    assert (pl["path"], pl["a_mode"], pl["bn"], pl["cta_pair"]) == (lib.PATH_WINDOW, 18, 128, 0)
    assert (pl["stages"], pl["weights_resident"], pl["tma_store"], pl["epilogue_c32"]) == (4, 1, 1, 0)
    assert (pl["tile_rows"], pl["m_tiles"], pl["k_blocks"]) == (112, 32 * 56 // 2, 3)
    # 128 channels at 56x56: a CTA pair with weight halves resident keeps four
    # slots with the full 64-column staging tile
    pl = lib.plan_info(128, 128, 56, 56, 128, 3, 3, 1, 1, 1)
    assert (pl["a_mode"], pl["cta_pair"], pl["stages"], pl["epilogue_c32"]) == (9, 1, 4, 0)
    # a one-row tile (W_out = 112) with 72 KB of weights: the ring's cap
    pl = lib.plan_info(128, 64, 112, 112, 64, 3, 3, 1, 1, 1)
    assert (pl["a_mode"], pl["bn"], pl["tile_rows"]) == (18, 64, 112) and pl["stages"] >= 7


def _window_smem_bytes(pl, shape):
    """Dynamic shared memory of a window-mode CTA, rebuilt from the plan's
    visible fields: header and alignment, B blocks (all of them when resident,
    KW per ring slot otherwise; half the columns on a CTA pair), the A slots of
    the staged rows, the pad that the last slot's reads of 128 + (KW-1)*d rows
    fall into, and the epilogue's staging tiles with the fp32 bias."""
    N, C_in, H, W, C_out, KH, KW, s, p, d = shape
    W_out = (W + 2 * p - (KW - 1) * d - 1) // s + 1
    wv = W_out + (KW - 1) * d
    rows = 128 // wv
    slot = -(-rows * wv * 128 // 1024) * 1024
    read = -(-(128 + (KW - 1) * d) // 8) * 8 * 128
    pad = max(0, read - slot)
    bnb = pl["bn"] // 2 if pl["cta_pair"] else pl["bn"]
    b_blocks = KH * KW * C_in // 64 if pl["weights_resident"] else pl["stages"] * KW
    if not pl["tma_store"]:
        epi = 0
    elif pl["epilogue_c32"]:
        epi = 8192 + 1024 + (pl["epilogue_tiles"] - 1) * 8192
    else:
        epi = 16384 + 1024 + (pl["epilogue_tiles"] - 1) * 16384
    return 512 + 1024 + b_blocks * bnb * 128 + pl["stages"] * slot + pad + epi, rows, W_out


def test_window_plans_fit_shared_memory(lib):
    # seeded random stride-1 shapes with C_in % 64 == 0: every plan the library
    # makes on the window path fits the 227 KB a CTA may hold, with its ring of
    # 2..8 slots and its tiles of whole output rows
    import random
    # the formula against a measured launch: ncu reports 229,888 bytes of dynamic
    # shared memory for the 64 -> 128 3x3 layer at 56x56 (four slots of 15 KB,
    # a 2 KB pad, 144 KB of weights, one staging tile)
    head = (32, 64, 56, 56, 128, 3, 3, 1, 1, 1)
    assert _window_smem_bytes(lib.plan_info(*head), head)[0] == 229888
    rng = random.Random(2024)
    seen, checked = set(), 0
    for _ in range(400):
        KH, KW = rng.choice([1, 2, 3, 5, 7]), rng.choice([2, 3, 5, 7])
        d = rng.choice([1, 1, 2])
        shape = (rng.choice([1, 2, 8, 32]), rng.choice([64, 128, 192, 256, 512]),
                 rng.randint(KH * d, 60), rng.randint(KW * d, 120),
                 rng.choice([32, 64, 96, 128, 192, 256, 384, 512]), KH, KW, 1,
                 rng.randint(0, (KW - 1) * d // 2 + 1), d)
        N, C_in, H, W, C_out = shape[:5]
        if lib.select_path(N, C_in, H, W, C_out, KH, KW, 1, shape[8], d) != lib.PATH_WINDOW:
            continue
        pl = lib.plan_info(*shape)
        if pl["a_mode"] not in (4, 9, 18):
            continue
        seen.add(pl["a_mode"])
        checked += 1
        smem, rows, W_out = _window_smem_bytes(pl, shape)
        assert smem <= 232448, (shape, pl, smem)
        assert 2 <= pl["stages"] <= 8, (shape, pl)
        assert pl["tile_rows"] == rows * W_out, (shape, pl)
        assert pl["k_blocks"] == KH * C_in // 64, (shape, pl)
    assert seen == {4, 9, 18} and checked >= 60, (seen, checked)


FOLD_GEOMS = [  # (N, H, W, C_out, KH, KW, pad, dilation)
    (1, 32, 32, 32, 3, 3, 1, 1), (3, 37, 45, 64, 3, 3, 1, 1), (2, 20, 70, 32, 5, 5, 2, 1),
    (1, 16, 40, 32, 7, 5, 3, 1), (2, 12, 33, 32, 3, 3, 2, 2), (4, 9, 64, 96, 3, 1, 1, 1),
    (2, 5, 64, 32, 1, 3, 1, 1), (1, 9, 40, 32, 3, 3, 5, 2), (8, 150, 150, 32, 3, 3, 1, 1),
]


@pytest.mark.parametrize("geom", FOLD_GEOMS, ids=str)
def test_winfold_plan_geometry(lib, geom):
    """The folded window's tiling, from the plan the library reports, against the
    geometry stated in include/convgb.h: segments of G = 32 - (KW-1)d output
    pixels, four output rows per tile, one tile per (image, row block,
    segment); 128- or 256-column accumulators by the MMA width KW*C_out; no
    workspace."""
    N, H, W, C_out, KH, KW, p, d = geom
    pl = lib.plan_info(N, 32, H, W, C_out, KH, KW, 1, p, d, path=lib.PATH_WINFOLD)
    Ho = oracle.output_size(H, KH, 1, p, d)
    Wo = oracle.output_size(W, KW, 1, p, d)
    G = 32 - (KW - 1) * d
    U = 8 if KH <= 3 and KW <= 3 and KW * C_out <= 128 else 4
    assert pl["segment_outputs"] == G and pl["tile_rows"] == 0 and pl["segment_rows"] == U
    assert pl["m_tiles"] == N * -(-Ho // U) * -(-Wo // G)
    assert pl["n_tiles"] == 1 and pl["splits"] == 1 and pl["k_blocks"] == 1
    assert pl["bn"] == (128 if KW * C_out <= 128 else 256)
    assert pl["a_mode"] == (17 if KH <= 3 and KW <= 3 else 16)
    # one stage per accumulator slot: four of 128 columns or two of 256, or two
    # pairs of 128 for 8-row units
    assert pl["stages"] == (2 if U == 8 else 4 if pl["bn"] == 128 else 2)
    if lib.select_path(N, 32, H, W, C_out, KH, KW, 1, p, d) == lib.PATH_WINFOLD:
        assert lib.workspace_size(N, 32, H, W, C_out, KH, KW, 1, p, d) == 0


def test_winfold_rejects_shapes_outside_its_limits(lib):
    for args in [(1, 32, 40, 40, 32, 3, 3, 2, 1, 1),    # stride 2
                 (1, 16, 40, 40, 32, 3, 3, 1, 1, 1),    # 16 channels
                 (1, 32, 31, 31, 32, 3, 3, 1, 1, 1),    # rows narrower than a segment
                 (1, 32, 40, 40, 48, 3, 3, 1, 1, 1),    # C_out not a multiple of 32
                 (1, 32, 40, 40, 64, 5, 5, 1, 2, 1),    # KW*C_out = 320 > 256
                 (1, 32, 40, 40, 32, 3, 3, 1, 13, 13),  # G = 6 < 8
                 (1, 32, 40, 40, 32, 9, 3, 1, 4, 1)]:   # KH = 9 > 7
        with pytest.raises(lib.ConvgbError):
            lib.plan_info(*args, path=lib.PATH_WINFOLD)


def test_dense_path_needs_no_workspace(lib):
    assert lib.workspace_size(32, 256, 56, 56, 64, 1, 1, 1, 0, 1) == 0
    assert lib.workspace_size(32, 512, 7, 7, 2048, 1, 1, 1, 0, 1) == 0


def test_split_k_only_for_underfilled_layers(lib):
    # full-spatial 7x7 -> 4096 at N=128: 16 output tiles, K split, fp32 sums [128][4096]
    assert lib.workspace_size(128, 512, 7, 7, 4096, 7, 7, 1, 0, 1) == 128 * 4096 * 4
    # the same 512-channel 7x7 layer on the gather path: 98 tiles, split;
    # ibuf (49*9*4 -> 1792 B) + sums.  The window path runs it as 64 CTA-pair
    # units, less than a wave of pairs, with no workspace; asked for stream-K,
    # its sums need the same [6272][512] fp32 buffer (12.8 MB, under half of the
    # 57.8 MB im2col)
    assert lib.workspace_size(128, 512, 7, 7, 512, 3, 3, 1, 1, 1, path=lib.PATH_GATHER) == \
        1792 + 6272 * 512 * 4
    assert lib.workspace_size(128, 512, 7, 7, 512, 3, 3, 1, 1, 1) == 0
    assert lib.plan_info(128, 512, 7, 7, 512, 3, 3, 1, 1, 1)["stream_k"] == 0
    lib.set_tuning(0, 0, 1)
    try:
        assert lib.workspace_size(128, 512, 7, 7, 512, 3, 3, 1, 1, 1) == 6272 * 512 * 4
        p = lib.plan_info(128, 512, 7, 7, 512, 3, 3, 1, 1, 1)
        assert p["stream_k"] == 1 and p["cta_pair"] == 1 and p["splits"] == 1
    finally:
        lib.set_tuning(0, 0, 0)
    # plenty of tiles: no split; the gather path needs only its indirection buffer
    assert lib.workspace_size(32, 64, 56, 56, 128, 3, 3, 1, 1, 1, path=lib.PATH_GATHER) == \
        56 * 56 * 9 * 4
    assert lib.workspace_size(32, 64, 56, 56, 128, 3, 3, 1, 1, 1) == 0
    # a split whose sums would not fit under half of im2col is not taken
    assert lib.workspace_size(5, 16, 5, 6, 130, 5, 6, 1, 0, 1) == 0
    # asking for the gather path on a 1x1 layer costs only the indirection buffer
    assert lib.workspace_size(32, 256, 56, 56, 64, 1, 1, 1, 0, 1, path=lib.PATH_GATHER) == \
        56 * 56 * 4


def test_path_support_matrix(lib):
    # stem path needs C_in % 8 != 0; gather and dense need C_in % 8 == 0
    assert lib.workspace_size(1, 3, 8, 8, 4, 3, 3, 1, 1, 1, path=lib.PATH_GATHER) == 0
    assert lib.workspace_size(1, 8, 8, 8, 4, 3, 3, 1, 1, 1, path=lib.PATH_STEM) == 0
    assert lib.workspace_size(1, 8, 8, 8, 4, 3, 3, 1, 1, 1, path=lib.PATH_DENSE) == 0
    assert lib.workspace_size(1, 3, 8, 8, 4, 3, 3, 1, 1, 1, path=lib.PATH_STEM) > 0


def call(lib, **kw):
    """Raw conv2d_fwd_path with fake (never dereferenced) pointers."""
    a = dict(path=0, x=0x1000, w=0x2000, b=0, N=1, C_in=8, H=8, W=8, C_out=8, KH=3, KW=3, s=1,
             p=1, d=1, y=0x3000, yd=0, ws=0x4000, wsb=1 << 20)
    a.update(kw)
    so = lib.load()
    P = ctypes.c_void_p
    return so.conv2d_fwd_path(a["path"], P(a["x"]), P(a["w"]), P(a["b"]), a["N"], a["C_in"],
                              a["H"], a["W"], a["C_out"], a["KH"], a["KW"], a["s"], a["p"],
                              a["d"], P(a["y"]), a["yd"], P(a["ws"]), a["wsb"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(N=0), 1), (dict(C_in=0), 1), (dict(KH=0), 1), (dict(s=0), 1), (dict(p=-1), 1),
    (dict(d=0), 1), (dict(H=2, p=0), 1), (dict(x=0), 1), (dict(w=0), 1), (dict(y=0), 1),
    (dict(yd=7), 1), (dict(path=9), 1), (dict(path=2), 2), (dict(path=3), 2), (dict(path=4), 2),
    (dict(wsb=16), 3), (dict(ws=0), 1), (dict(x=0x1008), 4), (dict(y=0x3004), 4),
    (dict(b=0x5002), 4), (dict(N=1 << 20, H=1 << 10, W=1 << 10), 2),
])
def test_bad_arguments_are_rejected_before_launch(lib, kw, status):
    assert call(lib, **kw) == status


def test_other_entry_points_reject_bad_arguments(lib):
    so = lib.load()
    P = ctypes.c_void_p
    assert so.build_indirection_buffer(8, 8, 8, 3, 3, 1, 1, 1, None, 1 << 20, None) == 1
    assert so.build_indirection_buffer(8, 8, 8, 3, 3, 1, 1, 1, P(0x1004), 1 << 20, None) == 4
    assert so.build_indirection_buffer(8, 8, 8, 3, 3, 1, 1, 1, P(0x1000), 16, None) == 3
    assert so.build_indirection_buffer(2, 2, 8, 3, 3, 1, 0, 1, P(0x1000), 1 << 20, None) == 1
    assert so.im2win_transform(None, 1, 8, 8, 8, 3, 3, 1, 1, 1, P(0x1000), 1 << 20, None) == 1
    assert so.im2win_transform(P(0x1000), 1, 8, 8, 8, 3, 3, 1, 1, 1, P(0x2000), 64, None) == 3
    assert so.im2win_transform(P(0x1002), 1, 8, 8, 8, 3, 3, 1, 1, 1, P(0x2000), 1 << 20, None) == 4


def test_host_entry_scratch_layout(lib):
    """conv2d_fwd_host's scratch: weights, bias, two input and two output slots of
    one chunk (the batch in up to four chunks of whole images), each rounded to
    256 bytes, plus the convolution workspace of the largest chunk."""
    r = lambda v: (v + 255) // 256 * 256

    def per_chunk(N):
        chunks = min(N, 4)
        return (N + chunks - 1) // chunks

    # N=32 -> 4 chunks of 8 images; the window path needs no workspace
    n = per_chunk(32)
    assert n == 8
    want = r(128 * 9 * 64 * 2) + r(128 * 2) + 2 * r(n * 56 * 56 * 64 * 2) + \
        2 * r(n * 56 * 56 * 128 * 2)
    assert lib.conv2d_fwd_host_scratch_size(32, 64, 56, 56, 128, 3, 3, 1, 1, 1) == want
    # no bias: no bias slot; fp32 output: output slots twice as large
    assert lib.conv2d_fwd_host_scratch_size(32, 64, 56, 56, 128, 3, 3, 1, 1, 1,
                                            has_bias=False) == want - r(256)
    import torch
    want32 = want + 2 * r(n * 56 * 56 * 128 * 4) - 2 * r(n * 56 * 56 * 128 * 2)
    assert lib.conv2d_fwd_host_scratch_size(32, 64, 56, 56, 128, 3, 3, 1, 1, 1,
                                            out_dtype=torch.float32) == want32
    # N=18 -> chunks of 5 images (four chunks, the last with three)
    n = per_chunk(18)
    assert n == 5
    assert lib.conv2d_fwd_host_scratch_size(18, 8, 6, 6, 8, 3, 3, 1, 1, 1) == \
        r(8 * 9 * 8 * 2) + r(16) + 2 * r(n * 36 * 8 * 2) + 2 * r(n * 36 * 8 * 2) + \
        r(max(lib.workspace_size(n, 8, 6, 6, 8, 3, 3, 1, 1, 1),
              lib.workspace_size(3, 8, 6, 6, 8, 3, 3, 1, 1, 1)))
    # invalid shapes have no scratch size
    assert lib.conv2d_fwd_host_scratch_size(1, 8, 2, 2, 8, 3, 3, 1, 0, 1) == 0
    assert lib.conv2d_fwd_host_scratch_size(0, 8, 8, 8, 8, 3, 3, 1, 1, 1) == 0


def test_host_entry_rejects_bad_arguments_before_cuda(lib):
    """No GPU here: every one of these must return before the first CUDA call."""
    so = lib.load()
    P = ctypes.c_void_p
    need = lib.conv2d_fwd_host_scratch_size(2, 8, 8, 8, 8, 3, 3, 1, 1, 1)

    def call(x=0x1000, w=0x2000, b=0x3000, y=0x4000, scratch=0x10000, nbytes=need, N=2,
             dtype=0, p=1):
        return so.conv2d_fwd_host(P(x) if x else None, P(w) if w else None,
                                  P(b) if b else None, N, 8, 8, 8, 8, 3, 3, 1, p, 1,
                                  P(y) if y else None, dtype, P(scratch) if scratch else None,
                                  nbytes, None)

    assert call(x=0) == 1
    assert call(w=0) == 1
    assert call(y=0) == 1
    assert call(scratch=0) == 1
    assert call(N=0) == 1
    assert call(dtype=7) == 1
    assert call(p=-1) == 1
    assert call(scratch=0x10008) == 4
    assert call(nbytes=need - 1) == 3
