"""GPU parity: every kernel, through the C ABI, against the CPU oracle.

Bars: the two re-layout kernels are compared bit for bit; the convolution
must satisfy, per element, |y - y_ref| <= 1e-2 * (|bias| + sum |x*w|) and, over
the tensor (or the sampled outputs), ||y - y_ref||_2 / ||y_ref||_2 <= 5e-3,
with y_ref the fp64 oracle on the same bf16 inputs.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL_ELEM = 1e-2
TOL_REL_L2 = 5e-3


def dev():
    return torch.device("cuda:0")


def check(got, ref, mag, what=""):
    got = np.asarray(got, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), what + ": non-finite output"
    err = np.abs(got - ref)
    bad = err > TOL_ELEM * mag
    assert not bad.any(), "%s: %d elements out of bound, worst err %.3g (bound %.3g)" % (
        what, bad.sum(), err[bad].max(), (TOL_ELEM * mag)[bad][np.argmax(err[bad])])
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / nref if nref > 0 else np.linalg.norm(got)
    assert rel <= TOL_REL_L2, "%s: relative L2 %.3g" % (what, rel)
    return err.max(), rel


def run_full(g, shape, path=0, out_dtype=torch.bfloat16, with_bias=True, seed=None):
    x, w, b = workloads.make_inputs(shape, seed=seed)
    if not with_bias:
        b = None
    y = g.conv2d_fwd_path(path, x.to(dev()), w.to(dev()), None if b is None else b.to(dev()),
                          shape.stride, shape.pad, shape.dilation, out_dtype=out_dtype)
    st, code = g.check_device_errors()
    assert st == 0, "device error word %#x" % code
    ref, mag = oracle.conv2d_direct(workloads.bits(x), workloads.bits(w),
                                    None if b is None else workloads.bits(b),
                                    shape.stride, shape.pad, shape.dilation)
    return y.float().cpu().numpy(), ref, mag


def S(name, **kw):
    d = dict(N=1, C_in=8, H=8, W=8, C_out=8, KH=3, KW=3, stride=1, pad=1, dilation=1, seed=11)
    d.update(kw)
    return workloads.ConvShape(name, **d)


# Small shapes that span several tiles, ragged M/N/K tails, every path and BN variant.
SMALL = [
    S("gather_3x3_ragged", N=2, C_in=16, H=13, W=11, C_out=24),
    S("gather_cout_100", N=1, C_in=64, H=15, W=17, C_out=100, seed=12),
    S("gather_cout_200", N=1, C_in=32, H=9, W=21, C_out=200, seed=13),
    S("gather_cout_300_k_tail", N=1, C_in=40, H=10, W=10, C_out=300, seed=14),
    S("gather_stride2_dil2", N=2, C_in=24, H=17, W=15, C_out=48, stride=2, pad=2, dilation=2, seed=15),
    S("gather_5x5_c96", N=1, C_in=96, H=12, W=12, C_out=64, KH=5, KW=5, pad=2, seed=16),
    S("gather_asym_kernel", N=3, C_in=8, H=9, W=14, C_out=16, KH=2, KW=4, stride=1, pad=1, seed=17),
    S("gather_1x1_pad", N=2, C_in=16, H=7, W=7, C_out=32, KH=1, KW=1, pad=1, seed=18),
    S("gather_1x1_s2", N=2, C_in=64, H=14, W=14, C_out=128, KH=1, KW=1, stride=2, pad=0, seed=19),
    S("dense_1x1", N=3, C_in=64, H=11, W=13, C_out=96, KH=1, KW=1, pad=0, seed=20),
    S("dense_1x1_ktail", N=2, C_in=72, H=9, W=9, C_out=40, KH=1, KW=1, pad=0, seed=21),
    S("dense_fullspatial", N=5, C_in=16, H=5, W=6, C_out=130, KH=5, KW=6, pad=0, seed=22),
    S("dense_fullspatial_splitk", N=8, C_in=64, H=7, W=7, C_out=200, KH=7, KW=7, pad=0, seed=28),
    S("gather_splitk_cout30", N=2, C_in=256, H=7, W=7, C_out=30, seed=29),
    S("gather_splitk_cout64", N=2, C_in=256, H=7, W=7, C_out=64, seed=30),
    S("tmagather_c128_s2_d2", N=2, C_in=128, H=17, W=15, C_out=96, stride=2, pad=2, dilation=2,
      seed=31),
    S("tmagather_c192_ragged", N=3, C_in=192, H=9, W=11, C_out=72, seed=32),
    S("tmagather_c64_5x3", N=2, C_in=64, H=12, W=13, C_out=256, KH=5, KW=3, pad=2, seed=33),
    S("window_c64_d2", N=2, C_in=64, H=20, W=21, C_out=48, pad=2, dilation=2, seed=34),
    S("window_c128_7x7_many_rows", N=3, C_in=128, H=7, W=7, C_out=64, seed=35),
    S("window_c64_cout200_streamed", N=2, C_in=64, H=11, W=13, C_out=200, seed=36),
    S("window_c64_5x5", N=1, C_in=64, H=16, W=18, C_out=32, KH=5, KW=5, pad=2, seed=37),
    S("window_c64_1x3", N=2, C_in=64, H=6, W=30, C_out=40, KH=1, KW=3, pad=1, seed=38),
    S("window_c64_wide_row", N=1, C_in=64, H=4, W=126, C_out=64, seed=39),
    S("stem_c3_7x7_s2", N=2, C_in=3, H=30, W=26, C_out=64, KH=7, KW=7, stride=2, pad=3, seed=23),
    S("stem_c1", N=2, C_in=1, H=12, W=12, C_out=16, seed=24),
    S("stem_c5", N=1, C_in=5, H=10, W=11, C_out=40, seed=25),
    S("stem_c12", N=1, C_in=12, H=9, W=9, C_out=32, KH=3, KW=3, seed=26),
    S("stem_11x11_s4", N=1, C_in=3, H=47, W=45, C_out=64, KH=11, KW=11, stride=4, pad=2, seed=27),
    # 1x1 stride > 1: element-strided TMA boxes (K tail, odd widths, stride 3, two column tiles)
    S("strided_1x1_s2_c72_ragged", N=3, C_in=72, H=10, W=13, C_out=96, KH=1, KW=1, stride=2,
      pad=0, seed=48),
    S("strided_1x1_s3_c16", N=2, C_in=16, H=17, W=20, C_out=40, KH=1, KW=1, stride=3, pad=0,
      seed=49),
    S("strided_1x1_s2_cout300", N=2, C_in=128, H=12, W=16, C_out=300, KH=1, KW=1, stride=2,
      pad=0, seed=50),
    # TMA gather on a CTA pair (256-wide column tiles): an odd tile count (the
    # last pair's second CTA gathers zeros) and two ragged column tiles
    S("tmagather_pair_c64_s2", N=4, C_in=64, H=18, W=20, C_out=256, stride=2, pad=1, seed=51),
    S("tmagather_pair_c128_cout300", N=8, C_in=128, H=11, W=9, C_out=300, stride=2, pad=1,
      seed=52),
    # window path on a CTA pair with 128-wide column tiles (weights too large to
    # stay resident on one CTA): resident halves, then streamed halves with an
    # odd tile count and a ragged column tile
    S("window_pair128_c128", N=3, C_in=128, H=12, W=12, C_out=128, seed=53),
    S("window_pair128_c192_cout100_odd", N=1, C_in=192, H=25, W=9, C_out=100, seed=54),
    # 32-column epilogue staging (64-byte swizzle), taken when it buys a ring
    # stage on tiles of at least 64 MMAs (a ragged last chunk in the second)
    S("window_c128_narrow_staging", N=1, C_in=128, H=30, W=30, C_out=128, seed=57),
    S("window_c128_cout120_narrow_staging", N=2, C_in=128, H=20, W=22, C_out=120, seed=58),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_conv_small_shapes_match_oracle(gpu_lib, shape, out_dtype):
    got, ref, mag = run_full(gpu_lib, shape, out_dtype=out_dtype)
    check(got, ref, mag, shape.name)


@pytest.mark.parametrize("shape", SMALL[:3] + SMALL[9:13], ids=lambda s: s.name)
def test_conv_without_bias(gpu_lib, shape):
    got, ref, mag = run_full(gpu_lib, shape, with_bias=False)
    check(got, ref, mag, shape.name)


# Shapes the window path takes (its geometry limits, and at most 6 weight
# blocks per ring slot when the weights are streamed).
WINDOW_ABLE = [sh for sh in SMALL if sh.stride == 1 and sh.C_in % 64 == 0 and
               (oracle.output_size(sh.W, sh.KW, 1, sh.pad, sh.dilation) +
                (sh.KW - 1) * sh.dilation) <= 128 and sh.KW <= 6]


@pytest.mark.parametrize("shape", WINDOW_ABLE, ids=lambda s: s.name)
@pytest.mark.parametrize("path", [1, 4], ids=["gather", "window"])
def test_window_and_gather_paths_match_oracle(gpu_lib, shape, path):
    """Both A producers on every shape the window path covers, explicitly."""
    got, ref, mag = run_full(gpu_lib, shape, path=path, out_dtype=torch.float32)
    check(got, ref, mag, shape.name)


# Plane path: the window path's shapes plus ones that reach its other plan
# choices: tiles that straddle images, two sub-tiles per weight block with a
# ragged column tile, split K, an output row of 128 padded pixels, and
# C_out % 8 != 0 (direct stores instead of the TMA-store epilogue).
PLANE_EXTRA = [
    S("plane_u2_c128_cout160", N=64, C_in=128, H=10, W=10, C_out=160, seed=40),
    S("plane_splitk_c512", N=1, C_in=512, H=5, W=6, C_out=64, seed=41),
    S("plane_cout30", N=3, C_in=64, H=9, W=10, C_out=30, seed=42),
    S("plane_c192_cout136", N=2, C_in=192, H=8, W=9, C_out=136, seed=43),
    S("plane_c64_5x3_d2", N=2, C_in=64, H=12, W=13, C_out=256, KH=5, KW=3, pad=2, dilation=2,
      seed=44),
]
PLANE_ABLE = WINDOW_ABLE + PLANE_EXTRA


@pytest.mark.parametrize("shape", PLANE_ABLE, ids=lambda s: s.name)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_plane_path_matches_oracle(gpu_lib, shape, out_dtype):
    got, ref, mag = run_full(gpu_lib, shape, path=gpu_lib.PATH_PLANE, out_dtype=out_dtype)
    check(got, ref, mag, shape.name)


# im2win path (small C_in): tiles of one or several output rows, a ragged last
# tile, streamed weights (C_out > 128), and 11x11 stride 4.
IM2WIN_SHAPES = [sh for sh in SMALL if sh.name in ("stem_c3_7x7_s2", "stem_c5", "stem_c12")] + [
    S("im2win_c3_11x11_s4", N=1, C_in=3, H=64, W=64, C_out=64, KH=11, KW=11, stride=4, pad=2,
      seed=45),
    S("im2win_c3_5x5_cout200", N=2, C_in=3, H=20, W=20, C_out=200, KH=5, KW=5, pad=2, seed=46),
    S("im2win_c7_7x7_s2", N=3, C_in=7, H=17, W=23, C_out=48, KH=7, KW=7, stride=2, pad=3,
      seed=47),
]
STEM_SHAPES = [sh for sh in SMALL if sh.C_in % 8 != 0]

# Staged-window stem (C_in = 3, stride 1/2/4): ragged last tile (7x7 s2), three
# kernel-row groups (11x11 s4) and two (9x9 s4), stride 1 (C_out not a multiple of
# 8 is excluded by the whole-copy rule of the raw weights), unpadded, and a
# 256-wide column tile; fp32 output takes the direct-store epilogue.
STEMWIN_SHAPES = [
    S("stemwin_c3_7x7_s2_ragged", N=3, C_in=3, H=29, W=32, C_out=64, KH=7, KW=7, stride=2,
      pad=3, seed=90),
    S("stemwin_c3_11x11_s4", N=2, C_in=3, H=64, W=64, C_out=64, KH=11, KW=11, stride=4, pad=2,
      seed=91),
    S("stemwin_c3_3x3_s1_cout40", N=2, C_in=3, H=16, W=16, C_out=40, seed=92),
    S("stemwin_c3_5x5_s2_cout40", N=2, C_in=3, H=20, W=24, C_out=40, KH=5, KW=5, stride=2, pad=2,
      seed=93),
    S("stemwin_c3_3x3_p0_cout128", N=2, C_in=3, H=10, W=16, C_out=128, pad=0, seed=94),
    S("stemwin_c3_3x3_s2_cout200", N=2, C_in=3, H=17, W=16, C_out=200, stride=2, seed=96),
    S("stemwin_c3_9x9_s4", N=1, C_in=3, H=48, W=48, C_out=32, KH=9, KW=9, stride=4, pad=4,
      seed=95),
]


@pytest.mark.parametrize("shape", STEMWIN_SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_stemwin_path_matches_oracle(gpu_lib, shape, out_dtype):
    plan = gpu_lib.plan_info(shape.N, shape.C_in, shape.H, shape.W, shape.C_out, shape.KH,
                             shape.KW, shape.stride, shape.pad, shape.dilation,
                             path=gpu_lib.PATH_STEMWIN)
    assert plan["a_mode"] in (13, 14, 15) and plan["stages"] >= 2, plan
    got, ref, mag = run_full(gpu_lib, shape, path=gpu_lib.PATH_STEMWIN, out_dtype=out_dtype)
    check(got, ref, mag, shape.name)


@pytest.mark.parametrize("shape", IM2WIN_SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_im2win_path_matches_oracle(gpu_lib, shape, out_dtype):
    got, ref, mag = run_full(gpu_lib, shape, path=gpu_lib.PATH_IM2WIN, out_dtype=out_dtype)
    check(got, ref, mag, shape.name)


@pytest.mark.parametrize("shape", STEM_SHAPES, ids=lambda s: s.name)
def test_stem_path_explicit_matches_oracle(gpu_lib, shape):
    """The staged-row and scalar stem kernels, which conv2d_fwd no longer picks
    where the im2win path applies."""
    got, ref, mag = run_full(gpu_lib, shape, path=gpu_lib.PATH_STEM, out_dtype=torch.float32)
    check(got, ref, mag, shape.name)


# Folded window (C_in = 32, stride 1): KW taps folded into the MMA's columns,
# the epilogue's shuffle sum across rows, padding columns left out of the sum.
# Ragged segments (W_out not a multiple of G), 64 output channels (192-column
# MMA), dilation 2 (G = 28, a row step of 2 in the segment's box), 5x5 and 7x5
# kernels (160-column MMA, KH up to 7), one kernel row, one kernel column with
# padding, no padding, rows exactly 32 pixels wide, and padding wider than the
# dilated kernel's reach into the image.
FOLD_SHAPES = [
    S("winfold_3x3_c32_ragged", N=2, C_in=32, H=9, W=37, C_out=32, seed=100),
    S("winfold_3x3_cout64", N=2, C_in=32, H=11, W=45, C_out=64, seed=101),
    S("winfold_3x3_d2", N=2, C_in=32, H=12, W=33, C_out=32, pad=2, dilation=2, seed=102),
    S("winfold_5x5_cout32", N=1, C_in=32, H=14, W=50, C_out=32, KH=5, KW=5, pad=2, seed=103),
    S("winfold_1x3", N=2, C_in=32, H=5, W=64, C_out=32, KH=1, KW=3, pad=1, seed=104),
    S("winfold_3x1_cout96", N=2, C_in=32, H=12, W=40, C_out=96, KH=3, KW=1, pad=1, seed=105),
    S("winfold_7x5", N=1, C_in=32, H=16, W=40, C_out=32, KH=7, KW=5, pad=3, seed=106),
    S("winfold_p0", N=3, C_in=32, H=8, W=70, C_out=32, pad=0, seed=107),
    S("winfold_w32_p2", N=2, C_in=32, H=6, W=32, C_out=32, pad=2, seed=108),
    S("winfold_d2_p5", N=1, C_in=32, H=9, W=40, C_out=32, pad=5, dilation=2, seed=109),
]


@pytest.mark.parametrize("shape", FOLD_SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_winfold_path_matches_oracle(gpu_lib, shape, out_dtype):
    plan = gpu_lib.plan_info(shape.N, shape.C_in, shape.H, shape.W, shape.C_out, shape.KH,
                             shape.KW, shape.stride, shape.pad, shape.dilation,
                             path=gpu_lib.PATH_WINFOLD)
    # kernels up to 3x3 take the instantiation with short tap loops
    small = shape.KH <= 3 and shape.KW <= 3
    assert plan["a_mode"] == (17 if small else 16) and plan["stages"] >= 2, plan
    assert plan["segment_outputs"] == 32 - (shape.KW - 1) * shape.dilation, plan
    got, ref, mag = run_full(gpu_lib, shape, path=gpu_lib.PATH_WINFOLD, out_dtype=out_dtype)
    check(got, ref, mag, shape.name)


@pytest.mark.parametrize("shape", FOLD_SHAPES[:2], ids=lambda s: s.name)
def test_winfold_without_bias(gpu_lib, shape):
    got, ref, mag = run_full(gpu_lib, shape, path=gpu_lib.PATH_WINFOLD, with_bias=False)
    check(got, ref, mag, shape.name)


def test_winfold_unaligned_output(gpu_lib):
    # y 16 bytes past a 32-byte boundary: the epilogue must not use 256-bit stores
    shape = FOLD_SHAPES[0]
    x, w, b = workloads.make_inputs(shape)
    Ho = oracle.output_size(shape.H, shape.KH, shape.stride, shape.pad, shape.dilation)
    Wo = oracle.output_size(shape.W, shape.KW, shape.stride, shape.pad, shape.dilation)
    n = shape.N * Ho * Wo * shape.C_out
    buf = torch.full((n + 16,), float("nan"), dtype=torch.bfloat16, device=dev())
    assert buf.data_ptr() % 32 == 0
    y = buf[8:8 + n].view(shape.N, Ho, Wo, shape.C_out)
    gpu_lib.conv2d_fwd_path(gpu_lib.PATH_WINFOLD, x.to(dev()), w.to(dev()), b.to(dev()),
                            shape.stride, shape.pad, shape.dilation, y=y)
    st, code = gpu_lib.check_device_errors()
    assert st == 0, "device error word %#x" % code
    ref, mag = oracle.conv2d_direct(workloads.bits(x), workloads.bits(w), workloads.bits(b),
                                    shape.stride, shape.pad, shape.dilation)
    check(y.float().cpu().numpy(), ref, mag, shape.name)
    assert torch.isnan(buf[:8].float()).all() and torch.isnan(buf[8 + n:].float()).all()


# One shape per A-operand mode whose grid hands every persistent CTA at least
# six work units (accumulator slots reused, the ring wrapped many times, pair
# tails at scale), with small K so the oracle checks every element in seconds.
MULTI_TILE = [
    (S("multi_gather_c32", N=130, C_in=32, H=30, W=30, C_out=32, seed=70), 1, 1),
    # folded window: two segments per 32-pixel output row (the second one
    # right-aligned in the row), then 64 output channels (192-column MMAs, two
    # 256-column accumulators)
    (S("multi_winfold_c32", N=130, C_in=32, H=30, W=32, C_out=32, seed=83), 0, 17),
    (S("multi_winfold_c32_cout64", N=64, C_in=32, H=30, W=40, C_out=64, seed=84), 8, 17),
    (S("multi_winfold_c32_5x5", N=64, C_in=32, H=30, W=40, C_out=32, KH=5, KW=5, pad=2,
       seed=85), 8, 16),
    (S("multi_tmagather_c64_s2", N=519, C_in=64, H=30, W=30, C_out=64, stride=2, seed=71), 0, 3),
    (S("multi_tmagather_pair_1x1_p1_s2", N=456, C_in=64, H=30, W=30, C_out=256, KH=1, KW=1,
       stride=2, pad=1, seed=72), 0, 12),
    (S("multi_window_pair_1x3", N=456, C_in=64, H=14, W=14, C_out=256, KH=1, KW=3, seed=73),
     0, 9),
    # (the window kernel built for the common plan: KW = 3, resident weights, TMA store)
    (S("multi_window_c64_1x3", N=456, C_in=64, H=14, W=14, C_out=64, KH=1, KW=3, seed=74), 0, 18),
    (S("multi_window_c64_1x5", N=456, C_in=64, H=14, W=14, C_out=64, KH=1, KW=5, pad=2, seed=86),
     0, 4),
    (S("multi_strided_1x1_s2", N=456, C_in=64, H=32, W=32, C_out=64, KH=1, KW=1, stride=2,
       pad=0, seed=75), 0, 11),
    (S("multi_dense_1x1", N=456, C_in=64, H=16, W=16, C_out=64, KH=1, KW=1, pad=0, seed=76),
     0, 0),
    # two column tiles, each CTA keeping its own column tile's weights resident
    (S("multi_strided_1x1_s2_cout512", N=228, C_in=64, H=32, W=32, C_out=512, KH=1, KW=1,
       stride=2, pad=0, seed=82), 0, 11),
    (S("multi_narrowwin_c3", N=114, C_in=3, H=32, W=32, C_out=32, seed=77), 3, 5),
    (S("multi_narrow_c3_d2", N=114, C_in=3, H=32, W=32, C_out=32, pad=2, dilation=2, seed=78),
     3, 2),
    (S("multi_im2win_c3_7x7_s2", N=456, C_in=3, H=32, W=32, C_out=64, KH=7, KW=7, stride=2,
       pad=3, seed=79), 6, 10),
    (S("multi_stemwin_c3_7x7_s2", N=456, C_in=3, H=32, W=32, C_out=64, KH=7, KW=7, stride=2,
       pad=3, seed=81), 7, 13),
    (S("multi_plane3_c64", N=456, C_in=64, H=14, W=14, C_out=64, seed=80), 5, None),
]


@pytest.mark.parametrize("case", MULTI_TILE, ids=lambda c: c[0].name)
def test_many_tiles_per_cta_every_element(gpu_lib, case):
    shape, path, amode = case
    plan = gpu_lib.plan_info(shape.N, shape.C_in, shape.H, shape.W, shape.C_out, shape.KH,
                             shape.KW, shape.stride, shape.pad, shape.dilation, path=path)
    if amode is not None:
        assert plan["a_mode"] == amode, plan
    units = plan["m_tiles"] * plan["n_tiles"] * plan["splits"]
    if plan["cta_pair"]:
        units = (plan["m_tiles"] + 1) // 2 * plan["n_tiles"]
        ctas = torch.cuda.get_device_properties(0).multi_processor_count // 2
    else:
        ctas = torch.cuda.get_device_properties(0).multi_processor_count
    assert units >= 6 * ctas, (units, ctas, plan)
    got, ref, mag = run_full(gpu_lib, shape, path=path)
    check(got, ref, mag, shape.name)


# Planner overrides used by the ablation study (convgb_set_tuning): forced tile
# widths and capped ring depths must still give exact results on every path.
TUNED_SHAPES = [sh for sh in SMALL if sh.name in (
    "gather_cout_200", "gather_cout_300_k_tail", "tmagather_c64_5x3", "dense_1x1",
    "window_c64_cout200_streamed", "window_c128_narrow_staging", "strided_1x1_s2_cout300",
    "stem_c3_7x7_s2", "stem_c5", "tmagather_pair_c128_cout300", "window_pair128_c128")] + [
    STEMWIN_SHAPES[0], STEMWIN_SHAPES[1]]
TUNINGS = [(32, 0), (64, 0), (128, 2), (256, 0), (0, 2), (0, 3)]


@pytest.fixture
def tuning(gpu_lib):
    yield gpu_lib.set_tuning
    gpu_lib.set_tuning(0, 0, 0)


@pytest.mark.parametrize("shape", TUNED_SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("bn,stages", TUNINGS, ids=lambda v: str(v))
def test_tuned_plans_match_oracle(gpu_lib, tuning, shape, bn, stages):
    tuning(bn, stages)
    plan = gpu_lib.plan_info(shape.N, shape.C_in, shape.H, shape.W, shape.C_out, shape.KH,
                             shape.KW, shape.stride, shape.pad, shape.dilation)
    if stages:
        # the TMA-gather modes never run on fewer than four stages; the
        # staged-window stem keeps the stages its raw weights pass through
        floor = 4 if plan["a_mode"] in (3, 12) else 2
        if plan["a_mode"] not in (13, 14, 15):
            assert plan["stages"] <= max(stages, floor)
        assert plan["stages"] >= floor
    got, ref, mag = run_full(gpu_lib, shape)
    check(got, ref, mag, "%s bn=%d stages<=%d" % (shape.name, bn, stages))


# Stream-K: units that fill less than a wave of CTA pairs share out all (unit,
# K block) steps equally; units cut between CTAs meet in fp32 partial sums.
STREAMK_SHAPES = [
    S("streamk_window_pair_c256_cout512_7x7", N=128, C_in=256, H=7, W=7, C_out=512, seed=85),
    S("streamk_window_pair_c128_cout160", N=64, C_in=128, H=10, W=10, C_out=160, seed=86),
]


@pytest.mark.parametrize("shape", STREAMK_SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_stream_k_matches_oracle(gpu_lib, tuning, shape, out_dtype):
    tuning(0, 0, 1)
    plan = gpu_lib.plan_info(shape.N, shape.C_in, shape.H, shape.W, shape.C_out, shape.KH,
                             shape.KW, shape.stride, shape.pad, shape.dilation,
                             out_dtype=out_dtype)
    assert plan["stream_k"] == 1, plan
    got, ref, mag = run_full(gpu_lib, shape, out_dtype=out_dtype)
    check(got, ref, mag, shape.name)


def test_tiny_config_full_output(gpu_lib):
    """3 -> 4 channels, 8x8, 3x3, fp32 output: every output element."""
    shape = workloads.TINY
    got, ref, mag = run_full(gpu_lib, shape, out_dtype=torch.float32)
    check(got, ref, mag, shape.name)


@pytest.mark.parametrize("shape", [SMALL[8], SMALL[9], SMALL[11]], ids=lambda s: s.name)
def test_paths_agree(gpu_lib, shape):
    """The gather path computes what the dense path computes (1x1 and full-spatial)."""
    x, w, b = workloads.make_inputs(shape)
    args = (x.to(dev()), w.to(dev()), b.to(dev()), shape.stride, shape.pad, shape.dilation)
    ys = {}
    for path in (gpu_lib.PATH_GATHER, gpu_lib.PATH_DENSE):
        try:
            ys[path] = gpu_lib.conv2d_fwd_path(path, *args, out_dtype=torch.float32)
        except gpu_lib.ConvgbError as e:
            assert e.status == 2  # dense path does not apply to this shape
    if len(ys) == 2:
        a, c = ys[gpu_lib.PATH_GATHER], ys[gpu_lib.PATH_DENSE]
        assert torch.allclose(a, c, rtol=1e-5, atol=1e-5)


def test_repeat_calls_are_deterministic(gpu_lib):
    shape = SMALL[1]
    x, w, b = workloads.make_inputs(shape)
    args = (x.to(dev()), w.to(dev()), b.to(dev()), shape.stride, shape.pad, shape.dilation)
    y1 = gpu_lib.conv2d_fwd(*args)
    y2 = gpu_lib.conv2d_fwd(*args)
    assert torch.equal(y1, y2)


def test_output_guard_bands_untouched(gpu_lib):
    """Writes stay inside y: canaries before and after the output survive."""
    shape = SMALL[3]
    x, w, b = workloads.make_inputs(shape)
    Ho = oracle.output_size(shape.H, shape.KH, shape.stride, shape.pad, shape.dilation)
    Wo = oracle.output_size(shape.W, shape.KW, shape.stride, shape.pad, shape.dilation)
    n = shape.N * Ho * Wo * shape.C_out
    guard = 4096
    buf = torch.full((n + 2 * guard,), 12345.0, dtype=torch.float32, device=dev())
    y = buf[guard:guard + n].view(shape.N, Ho, Wo, shape.C_out)
    gpu_lib.conv2d_fwd(x.to(dev()), w.to(dev()), b.to(dev()), shape.stride, shape.pad,
                       shape.dilation, out_dtype=torch.float32, y=y)
    torch.cuda.synchronize()
    assert torch.all(buf[:guard] == 12345.0) and torch.all(buf[guard + n:] == 12345.0)


INDIR_GEOMS = [(8, 8, 8, 3, 3, 1, 1, 1), (13, 11, 16, 3, 3, 2, 1, 1), (56, 56, 64, 3, 3, 1, 1, 1),
               (224, 224, 3, 7, 7, 2, 3, 1), (28, 28, 256, 3, 3, 1, 2, 2),
               (27, 27, 96, 5, 5, 1, 2, 1), (224, 224, 3, 11, 11, 4, 2, 1), (7, 7, 512, 7, 7, 1, 0, 1),
               (9, 14, 8, 2, 4, 3, 3, 2)]


@pytest.mark.parametrize("geom", INDIR_GEOMS, ids=str)
def test_indirection_buffer_bit_exact(gpu_lib, geom):
    H, W, C, KH, KW, s, p, d = geom
    got = gpu_lib.build_indirection_buffer(H, W, C, KH, KW, s, p, d, device=dev()).cpu().numpy()
    ref = oracle.indirection_buffer(H, W, C, KH, KW, s, p, d)
    np.testing.assert_array_equal(got, ref)


IM2WIN = [S("w_3x3", N=2, C_in=16, H=9, W=10), S("w_s2d2", N=2, C_in=8, H=17, W=15, stride=2, pad=2,
                                                dilation=2),
          S("w_5x5_c96", N=1, C_in=96, H=12, W=12, KH=5, KW=5, pad=2),
          S("w_c3_7x7", N=2, C_in=3, H=30, W=26, KH=7, KW=7, stride=2, pad=3),
          S("w_c5", N=1, C_in=5, H=10, W=11), S("w_resnet", N=4, C_in=64, H=56, W=56)]


@pytest.mark.parametrize("shape", IM2WIN, ids=lambda s: s.name)
def test_im2win_bit_exact(gpu_lib, shape):
    x, _, _ = workloads.make_inputs(shape)
    win = gpu_lib.im2win_transform(x.to(dev()), shape.KH, shape.KW, shape.stride, shape.pad,
                                   shape.dilation)
    got = win.cpu().view(torch.int16).numpy().view(np.uint16)
    ref = oracle.im2win(workloads.bits(x), shape.KH, shape.KW, shape.stride, shape.pad,
                        shape.dilation)
    np.testing.assert_array_equal(got, ref)


def test_wait_timeout_is_reported_not_hung(gpu_lib):
    """A wait nothing satisfies gives up after its limit and reports INTERNAL."""
    st, _ = gpu_lib.check_device_errors()
    assert st == 0
    gpu_lib.selftest_wait_timeout(2_000_000)  # 2 ms
    st, code = gpu_lib.check_device_errors()
    assert st == gpu_lib.ERR_INTERNAL
    assert code & 0xFF == 1 and (code >> 8) == 5
    # the context stays usable and the word is cleared
    st, _ = gpu_lib.check_device_errors()
    assert st == 0
    got, ref, mag = run_full(gpu_lib, SMALL[0])
    check(got, ref, mag, "after timeout")


def test_dependent_layers_back_to_back(gpu_lib):
    """A chain of layers on one stream with no host synchronisation: each layer
    reads the previous layer's output and overwrites the buffer the layer
    before it read.  The convolution kernel may start on SMs the previous
    kernel has left (programmatic stream serialization) and must wait for that
    kernel before touching global memory, so the chain must equal, bit for bit,
    the same chain run with a full synchronisation after every layer (no split
    K here: every output element has one fixed reduction order)."""
    g = gpu_lib
    x, _, _ = workloads.make_inputs(S("chain_x", N=2, C_in=64, H=14, W=14, C_out=64, seed=55))
    layers = []
    for i, (k, path) in enumerate([(3, 0), (1, 0), (3, g.PATH_GATHER), (3, 0)]):
        sh = S("chain%d" % i, N=2, C_in=64, H=14, W=14, C_out=64, KH=k, KW=k, pad=k // 2,
               seed=56 + i)
        _, w, b = workloads.make_inputs(sh)
        layers.append((sh, path, w.to(dev()), b.to(dev())))

    def run(sync):
        src = x.to(dev()).clone()
        dst = torch.empty_like(src)
        outs = []
        for _ in range(3):
            for sh, path, w, b in layers:
                g.conv2d_fwd_path(path, src, w, b, sh.stride, sh.pad, sh.dilation, y=dst)
                if sync:
                    torch.cuda.synchronize()
                    outs.append(dst.cpu())
                src, dst = dst, src
        torch.cuda.synchronize()
        st, code = g.check_device_errors()
        assert st == 0, "device error word %#x" % code
        return src.cpu(), outs

    chained, _ = run(False)
    stepped, outs = run(True)
    assert torch.equal(chained.view(torch.int16), stepped.view(torch.int16))
    # the synchronised chain's last layer against the oracle on its own input
    sh, path, w, b = layers[-1]
    ref, mag = oracle.conv2d_direct(workloads.bits(outs[-2]), workloads.bits(w.cpu()),
                                    workloads.bits(b.cpu()), sh.stride, sh.pad, sh.dilation)
    check(outs[-1].float().numpy(), ref, mag, "chain, last layer")


HOST_SHAPES = [
    # three chunks of 2, 2 and 1 images on the window path
    S("host_window_n5", N=5, C_in=64, H=12, W=12, C_out=64, seed=61),
    # the stem (im2win path, whose workspace is per chunk), fp32 output
    S("host_stem_n3", N=3, C_in=3, H=20, W=22, C_out=16, KH=7, KW=7, stride=2, pad=3, seed=62),
    # four chunks of one image, 1x1
    S("host_dense_n4", N=4, C_in=32, H=9, W=7, C_out=40, KH=1, KW=1, pad=0, seed=63),
    # four chunks of 5 images: each of the two slots is reused
    S("host_window_n20", N=20, C_in=64, H=10, W=10, C_out=64, seed=64),
]


@pytest.mark.parametrize("shape", HOST_SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_buffers_match_oracle(gpu_lib, shape, pinned):
    """conv2d_fwd_host: inputs read from and output written to host memory, the
    batch pipelined in chunks; y is valid once the stream has finished."""
    g = gpu_lib
    x, w, b = workloads.make_inputs(shape)
    out_dtype = torch.float32 if "stem" in shape.name else torch.bfloat16
    y = None
    if pinned:
        x, w, b = x.pin_memory(), w.pin_memory(), b.pin_memory()
    else:
        ho, wo = g.output_dims(shape.H, shape.W, shape.KH, shape.KW, shape.stride, shape.pad,
                               shape.dilation)
        y = torch.empty((shape.N, ho, wo, shape.C_out), dtype=out_dtype)
    y = g.conv2d_fwd_host(x, w, b, shape.stride, shape.pad, shape.dilation, out_dtype=out_dtype,
                          y=y)
    torch.cuda.current_stream().synchronize()
    st, code = g.check_device_errors()
    assert st == 0, "device error word %#x" % code
    ref, mag = oracle.conv2d_direct(workloads.bits(x), workloads.bits(w), workloads.bits(b),
                                    shape.stride, shape.pad, shape.dilation)
    check(y.float().numpy(), ref, mag, shape.name)


def test_host_buffers_without_bias(gpu_lib):
    shape = HOST_SHAPES[0]
    x, w, _ = workloads.make_inputs(shape)
    y = gpu_lib.conv2d_fwd_host(x.pin_memory(), w.pin_memory(), None, shape.stride, shape.pad,
                                shape.dilation)
    torch.cuda.current_stream().synchronize()
    ref, mag = oracle.conv2d_direct(workloads.bits(x), workloads.bits(w), None, shape.stride,
                                    shape.pad, shape.dilation)
    check(y.float().numpy(), ref, mag, "host, no bias")
