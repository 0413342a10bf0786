"""conv2d_fwd_noalloc, the entry point for callers that cannot provide a workspace.

Some callers cannot allocate device memory for the library: their memory is
planned by a host framework with no allocation hook, or they run loops that
must never call cudaMalloc/cudaFree.  conv2d_fwd_noalloc keeps its scratch
(the indirection buffer) in a fixed array inside the library instead.  These
tests call it through the C ABI and check that it reproduces conv2d_fwd,
within the parity tolerances, on consecutive calls that reuse that array with
different shapes.  The file sorts last so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from test_gpu_parity import TOL_ELEM, TOL_REL_L2

pytestmark = pytest.mark.gpu


def noalloc(g, x, w, b, shape, y, f32):
    P = ctypes.c_void_p
    return g.load().conv2d_fwd_noalloc(
        P(x.data_ptr()), P(w.data_ptr()), None if b is None else P(b.data_ptr()),
        shape.N, shape.C_in, shape.H, shape.W, shape.C_out, shape.KH, shape.KW, shape.stride,
        shape.pad, shape.dilation, P(y.data_ptr()), 1 if f32 else 0,
        P(torch.cuda.current_stream().cuda_stream))


SHAPES = [
    workloads.ConvShape("noalloc_3x3", N=2, C_in=32, H=19, W=17, C_out=96, KH=3, KW=3, pad=1,
                        seed=41),
    workloads.ConvShape("noalloc_5x5_s2_d1", N=1, C_in=16, H=23, W=29, C_out=40, KH=5, KW=5,
                        stride=2, pad=2, seed=42),
    workloads.ConvShape("noalloc_3x3_again", N=2, C_in=32, H=19, W=17, C_out=96, KH=3, KW=3,
                        pad=1, seed=43),
]


def test_noalloc_matches_conv2d_fwd_on_consecutive_calls(gpu_lib):
    dev = torch.device("cuda:0")
    for i, shape in enumerate(SHAPES):
        f32 = i == 1
        x, w, b = workloads.make_inputs(shape)
        xd, wd, bd = x.to(dev), w.to(dev), b.to(dev)
        out_dtype = torch.float32 if f32 else torch.bfloat16
        y_ref = gpu_lib.conv2d_fwd(xd, wd, bd, shape.stride, shape.pad, shape.dilation,
                                   out_dtype=out_dtype)
        y = torch.full_like(y_ref, float("nan"))
        assert noalloc(gpu_lib, xd, wd, bd, shape, y, f32) == 0
        st, code = gpu_lib.check_device_errors()
        assert st == 0, "device error word %#x" % code
        _, mag = oracle.conv2d_direct(workloads.bits(x), workloads.bits(w), workloads.bits(b),
                                      shape.stride, shape.pad, shape.dilation)
        got = y.double().cpu().numpy()
        ref = y_ref.double().cpu().numpy()
        assert np.all(np.isfinite(got))
        assert np.all(np.abs(got - ref) <= TOL_ELEM * mag), shape.name
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel <= TOL_REL_L2, (shape.name, rel)


def test_noalloc_rejects_shapes_beyond_its_scratch(gpu_lib):
    # 600x600 output, 3x3 taps: 3.24M indirection entries > the 1,048,576 the array holds
    shape = workloads.ConvShape("too_big", N=1, C_in=8, H=600, W=600, C_out=8, KH=3, KW=3,
                                pad=1)
    dev = torch.device("cuda:0")
    x = torch.zeros((1, 600, 600, 8), dtype=torch.bfloat16, device=dev)
    w = torch.zeros((8, 3, 3, 8), dtype=torch.bfloat16, device=dev)
    y = torch.zeros((1, 600, 600, 8), dtype=torch.bfloat16, device=dev)
    assert noalloc(gpu_lib, x, w, None, shape, y, False) == 3  # CONVGB_ERR_WORKSPACE
    c3 = workloads.ConvShape("c3", N=1, C_in=3, H=8, W=8, C_out=8, KH=3, KW=3, pad=1)
    x3 = torch.zeros((1, 8, 8, 3), dtype=torch.bfloat16, device=dev)
    w3 = torch.zeros((8, 3, 3, 3), dtype=torch.bfloat16, device=dev)
    y3 = torch.zeros((1, 8, 8, 8), dtype=torch.bfloat16, device=dev)
    assert noalloc(gpu_lib, x3, w3, None, c3, y3, False) == 2  # gather path only
    torch.cuda.synchronize()
