"""GPU parity at the full benchmark sizes, in the launch configuration the
benchmark times (conv2d_fwd on the library's own path choice).

The five configurations of the tiny, ResNet-style, 1x1 and stem groups are
checked on every output element against the fp64 oracle (seconds of CPU work
each).  The N=128 layer sweep is checked on outputs drawn per tile of the plan
the library launches (convgb_plan_info): several points in every (row tile,
column tile) pair, so no tile of the persistent kernel's loop goes unchecked,
plus the corners and borders of the first and last image, where padding
matters.  The explicit plane and stem paths at full size are checked the same
way.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from test_gpu_parity import TOL_ELEM, TOL_REL_L2, check

pytestmark = pytest.mark.gpu

PER_TILE = 4


def border_points(shape, Ho, Wo):
    pts = []
    for n in (0, shape.N - 1):
        for ho in (0, Ho - 1):
            for wo in (0, Wo - 1):
                for co in (0, shape.C_out - 1):
                    pts.append((n, co, ho, wo))
        for ho in range(Ho):  # left and right borders
            pts.append((n, ho % shape.C_out, ho, 0))
            pts.append((n, (ho + 1) % shape.C_out, ho, Wo - 1))
        for wo in range(Wo):  # top and bottom borders
            pts.append((n, wo % shape.C_out, 0, wo))
            pts.append((n, (wo + 1) % shape.C_out, Ho - 1, wo))
    return np.array(pts, dtype=np.int64)


def fold_tile_points(shape, plan, Ho, Wo, rng, per_tile=PER_TILE):
    """Folded-window plans: tile t = (n*HB + hb)*spr + k holds output pixels
    k*G .. k*G + G - 1 (G = segment_outputs, spr segments per row, the last one
    shorter) of output rows U*hb .. U*hb + U - 1 (U = segment_rows, HB =
    ceil(H_out / U) row blocks).  per_tile / 4 (at least one) random outputs in
    each of a tile's rows."""
    G, U = plan["segment_outputs"], plan["segment_rows"]
    spr = -(-Wo // G)
    HB = -(-Ho // U)
    assert plan["m_tiles"] == shape.N * HB * spr, plan
    per_row = max(1, per_tile // 4)
    t = np.repeat(np.arange(plan["m_tiles"], dtype=np.int64), U * per_row)
    q = np.tile(np.repeat(np.arange(U, dtype=np.int64), per_row), plan["m_tiles"])
    nhb, k = np.divmod(t, spr)
    n, hb = np.divmod(nhb, HB)
    ho = hb * U + q
    keep = ho < Ho
    t, k, n, ho = t[keep], k[keep], n[keep], ho[keep]
    span = np.minimum(Wo, (k + 1) * G) - k * G
    wo = k * G + (rng.random(len(t)) * span).astype(np.int64)
    co = rng.integers(0, shape.C_out, len(t))
    return np.stack([n, co, ho, wo], axis=1)


def tile_points(shape, plan, Ho, Wo, rng, per_tile=PER_TILE):
    """per_tile random outputs inside every (row tile, column tile) of the plan."""
    if plan.get("segment_outputs", 0):
        return fold_tile_points(shape, plan, Ho, Wo, rng, per_tile)
    M = shape.N * Ho * Wo
    tr = plan["tile_rows"]
    assert tr > 0, "the plan's tiles are not ranges of M"
    mt = np.repeat(np.arange(plan["m_tiles"], dtype=np.int64), plan["n_tiles"] * per_tile)
    nt = np.tile(np.repeat(np.arange(plan["n_tiles"], dtype=np.int64), per_tile), plan["m_tiles"])
    lo = mt * tr
    span = np.minimum(M, lo + tr) - lo
    assert np.all(span > 0), "a row tile lies past the end of M"
    m = lo + (rng.random(len(mt)) * span).astype(np.int64)
    c_lo = nt * plan["bn"]
    c_span = np.minimum(shape.C_out, c_lo + plan["bn"]) - c_lo
    co = c_lo + (rng.random(len(nt)) * c_span).astype(np.int64)
    n, pix = np.divmod(m, Ho * Wo)
    ho, wo = np.divmod(pix, Wo)
    return np.stack([n, co, ho, wo], axis=1)


def run_conv(gpu_lib, shape, path):
    x, w, b = workloads.make_inputs(shape)
    d = torch.device("cuda:0")
    out_dtype = torch.float32 if shape.out_f32 else torch.bfloat16
    y = gpu_lib.conv2d_fwd_path(path, x.to(d), w.to(d), b.to(d), shape.stride, shape.pad,
                                shape.dilation, out_dtype=out_dtype)
    st, code = gpu_lib.check_device_errors()
    assert st == 0, "device error word %#x" % code
    Ho, Wo = y.shape[1], y.shape[2]
    assert Ho == oracle.output_size(shape.H, shape.KH, shape.stride, shape.pad, shape.dilation)
    assert Wo == oracle.output_size(shape.W, shape.KW, shape.stride, shape.pad, shape.dilation)
    return x, w, b, y


# configs of the tiny, ResNet-style, 1x1 and stem groups: every output element
WHOLE = [c for g in ("tiny", "resnet3x3", "pointwise", "stem") for c in workloads.GROUPS[g]]


@pytest.mark.parametrize("shape", WHOLE, ids=lambda s: s.name)
def test_full_size_config_every_element(gpu_lib, shape):
    x, w, b, y = run_conv(gpu_lib, shape, 0)
    ref, mag = oracle.conv2d_direct(workloads.bits(x), workloads.bits(w), workloads.bits(b),
                                    shape.stride, shape.pad, shape.dilation)
    check(y.float().cpu().numpy(), ref, mag, shape.name)


def check_per_tile(gpu_lib, shape, path, per_tile=PER_TILE):
    out_dtype = torch.float32 if shape.out_f32 else torch.bfloat16
    plan = gpu_lib.plan_info(shape.N, shape.C_in, shape.H, shape.W, shape.C_out, shape.KH,
                             shape.KW, shape.stride, shape.pad, shape.dilation, path=path,
                             out_dtype=out_dtype)
    x, w, b, y = run_conv(gpu_lib, shape, path)
    Ho, Wo = y.shape[1], y.shape[2]
    rng = np.random.default_rng(shape.seed)
    pts = np.concatenate([border_points(shape, Ho, Wo),
                          tile_points(shape, plan, Ho, Wo, rng, per_tile)])
    ref, mag = oracle.conv2d_points(workloads.bits(x), workloads.bits(w), workloads.bits(b),
                                    shape.stride, shape.pad, shape.dilation, pts)
    yc = y.float().cpu().numpy()
    got = yc[pts[:, 0], pts[:, 2], pts[:, 3], pts[:, 1]].astype(np.float64)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    bad = err > TOL_ELEM * mag
    assert not bad.any(), "%s: %d of %d sampled outputs out of bound (worst %.3g)" % (
        shape.name, bad.sum(), len(pts), err.max())
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= TOL_REL_L2, rel
    return plan, len(pts)


@pytest.mark.parametrize("shape", workloads.SWEEP, ids=lambda s: s.name)
def test_sweep_every_tile_sampled(gpu_lib, shape):
    # the full-spatial layer has one row tile: more points per column tile
    per = 32 if shape.KH == shape.H else PER_TILE
    check_per_tile(gpu_lib, shape, 0, per)


def plane_able(c):
    return (c.stride == 1 and c.C_in % 64 == 0 and c.W + 2 * c.pad <= 128 and
            (c.KW - 1) * c.dilation <= 8)


FULL = [c for c in workloads.ALL if c.name != workloads.TINY.name]


@pytest.mark.parametrize("shape", [c for c in FULL if plane_able(c)], ids=lambda s: s.name)
def test_full_size_plane_path_sampled(gpu_lib, shape):
    # plane tiles hold padding-border pixels and are not ranges of M: the
    # per-tile draw runs on the output rows instead (every output row of
    # every image gets points)
    x, w, b, y = run_conv(gpu_lib, shape, gpu_lib.PATH_PLANE)
    Ho, Wo = y.shape[1], y.shape[2]
    rng = np.random.default_rng(shape.seed)
    rows = np.repeat(np.arange(shape.N * Ho, dtype=np.int64), 2)
    n, ho = np.divmod(rows, Ho)
    wo = rng.integers(0, Wo, len(rows))
    co = rng.integers(0, shape.C_out, len(rows))
    pts = np.concatenate([border_points(shape, Ho, Wo), np.stack([n, co, ho, wo], axis=1)])
    ref, mag = oracle.conv2d_points(workloads.bits(x), workloads.bits(w), workloads.bits(b),
                                    shape.stride, shape.pad, shape.dilation, pts)
    yc = y.float().cpu().numpy()
    got = yc[pts[:, 0], pts[:, 2], pts[:, 3], pts[:, 1]].astype(np.float64)
    err = np.abs(got - ref)
    assert not (err > TOL_ELEM * mag).any(), shape.name
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= TOL_REL_L2


@pytest.mark.parametrize("shape", [c for c in FULL if c.C_in == 32], ids=lambda s: s.name)
def test_full_size_gather_path_for_32_channels_sampled(gpu_lib, shape):
    """The gather path, which conv2d_fwd no longer picks for 32-channel layers
    the folded window takes, at full size."""
    check_per_tile(gpu_lib, shape, gpu_lib.PATH_GATHER)


@pytest.mark.parametrize("shape", [c for c in FULL if c.C_in % 8 != 0], ids=lambda s: s.name)
@pytest.mark.parametrize("path", ["stem", "im2win"])
def test_full_size_other_stem_paths_sampled(gpu_lib, shape, path):
    """The staged-row and im2win paths, which conv2d_fwd no longer picks for
    these layers, at full size."""
    check_per_tile(gpu_lib, shape, gpu_lib.PATH_STEM if path == "stem" else gpu_lib.PATH_IM2WIN)
