"""GPU parity at the full benchmark sizes, in the launch configuration the
benchmark times (conv2d_fwd on the library's own path choice).

The oracle computes a seeded sample of output elements one by one (every
output is too slow on the CPU at these sizes); the sample always includes
the four image corners and border pixels of the first and last image, where
padding matters, plus uniformly drawn interior points.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from test_gpu_parity import TOL_ELEM, TOL_REL_L2

pytestmark = pytest.mark.gpu

SAMPLES = 1500


def sample_points(shape, Ho, Wo, rng):
    pts = []
    for n in (0, shape.N - 1):
        for ho in (0, Ho - 1):
            for wo in (0, Wo - 1):
                for co in (0, shape.C_out - 1):
                    pts.append((n, co, ho, wo))
    k = SAMPLES - len(pts)
    pts += list(zip(rng.integers(0, shape.N, k), rng.integers(0, shape.C_out, k),
                    rng.integers(0, Ho, k), rng.integers(0, Wo, k)))
    return np.array(pts, dtype=np.int64)


def plane_able(c):
    return (c.stride == 1 and c.C_in % 64 == 0 and c.W + 2 * c.pad <= 128 and
            (c.KW - 1) * c.dilation <= 8)


FULL = [c for c in workloads.ALL if c.name != workloads.TINY.name]


@pytest.mark.parametrize("shape", FULL, ids=lambda s: s.name)
def test_full_size_config_sampled(gpu_lib, shape):
    check_sampled(gpu_lib, shape, 0)


@pytest.mark.parametrize("shape", [c for c in FULL if plane_able(c)], ids=lambda s: s.name)
def test_full_size_plane_path_sampled(gpu_lib, shape):
    check_sampled(gpu_lib, shape, gpu_lib.PATH_PLANE)


@pytest.mark.parametrize("shape", [c for c in FULL if c.C_in % 8 != 0], ids=lambda s: s.name)
def test_full_size_stem_path_sampled(gpu_lib, shape):
    check_sampled(gpu_lib, shape, gpu_lib.PATH_STEM)


def check_sampled(gpu_lib, shape, path):
    x, w, b = workloads.make_inputs(shape)
    d = torch.device("cuda:0")
    out_dtype = torch.float32 if shape.out_f32 else torch.bfloat16
    y = gpu_lib.conv2d_fwd_path(path, x.to(d), w.to(d), b.to(d), shape.stride, shape.pad,
                                shape.dilation, out_dtype=out_dtype)
    st, code = gpu_lib.check_device_errors()
    assert st == 0, "device error word %#x" % code
    assert bool(torch.isfinite(y).all())
    Ho, Wo = y.shape[1], y.shape[2]
    assert Ho == oracle.output_size(shape.H, shape.KH, shape.stride, shape.pad, shape.dilation)
    assert Wo == oracle.output_size(shape.W, shape.KW, shape.stride, shape.pad, shape.dilation)
    pts = sample_points(shape, Ho, Wo, np.random.default_rng(shape.seed))
    ref, mag = oracle.conv2d_points(workloads.bits(x), workloads.bits(w), workloads.bits(b),
                                    shape.stride, shape.pad, shape.dilation, pts)
    yc = y.float().cpu().numpy()
    got = yc[pts[:, 0], pts[:, 2], pts[:, 3], pts[:, 1]].astype(np.float64)
    err = np.abs(got - ref)
    bad = err > TOL_ELEM * mag
    assert not bad.any(), "%d of %d sampled outputs out of bound (worst %.3g)" % (
        bad.sum(), len(pts), err.max())
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= TOL_REL_L2, rel
