"""conv2d_fwd_noalloc, the entry point for callers that cannot provide a workspace.

Some callers cannot allocate device memory for the library: their memory is
planned by a host framework with no allocation hook, or they run loops that
must never call cudaMalloc/cudaFree.  conv2d_fwd_noalloc keeps its scratch
(the indirection buffer) in a fixed array inside the library instead.  These
tests call it through the C ABI and check its output against the fp64 oracle,
within the parity tolerances, on consecutive calls that reuse that array with
different shapes: the 16-byte cp.async gather, the TMA gather on one CTA and
on a CTA pair (256-wide column tiles), and a small layer whose conv2d_fwd plan
would split K (this entry point never splits: it has nowhere to keep partial
sums).  The last call repeats the first shape, so the array's previous
contents are another shape's.  The file sorts last so that a run stopping at
the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import oracle
import workloads
from test_gpu_parity import check

pytestmark = pytest.mark.gpu


def noalloc(g, x, w, b, shape, y, f32):
    P = ctypes.c_void_p
    return g.load().conv2d_fwd_noalloc(
        P(x.data_ptr()), P(w.data_ptr()), None if b is None else P(b.data_ptr()),
        shape.N, shape.C_in, shape.H, shape.W, shape.C_out, shape.KH, shape.KW, shape.stride,
        shape.pad, shape.dilation, P(y.data_ptr()), 1 if f32 else 0,
        P(torch.cuda.current_stream().cuda_stream))


def S(name, **kw):
    return workloads.ConvShape(name, **kw)


# (shape, fp32 output, kernel A mode the gather plan uses)
CASES = [
    (S("noalloc_3x3_c32", N=2, C_in=32, H=19, W=17, C_out=96, KH=3, KW=3, pad=1, seed=41),
     False, 1),
    (S("noalloc_5x5_s2_c16", N=1, C_in=16, H=23, W=29, C_out=40, KH=5, KW=5, stride=2, pad=2,
       seed=42), True, 1),
    (S("noalloc_tmagather_pair_c64_cout256", N=2, C_in=64, H=20, W=20, C_out=256, KH=3, KW=3,
       pad=1, seed=44), False, 12),
    (S("noalloc_small_m_c256", N=2, C_in=256, H=7, W=7, C_out=64, KH=3, KW=3, pad=1, seed=45),
     False, 3),
    (S("noalloc_3x3_c32_again", N=2, C_in=32, H=19, W=17, C_out=96, KH=3, KW=3, pad=1, seed=43),
     False, 1),
]


def test_noalloc_matches_oracle_on_consecutive_calls(gpu_lib):
    dev = torch.device("cuda:0")
    # the small-M case really is one whose conv2d_fwd plan splits K
    sm = CASES[3][0]
    assert gpu_lib.plan_info(sm.N, sm.C_in, sm.H, sm.W, sm.C_out, sm.KH, sm.KW, sm.stride,
                             sm.pad, sm.dilation, path=gpu_lib.PATH_GATHER)["splits"] > 1
    for shape, f32, amode in CASES:
        plan = gpu_lib.plan_info(shape.N, shape.C_in, shape.H, shape.W, shape.C_out, shape.KH,
                                 shape.KW, shape.stride, shape.pad, shape.dilation,
                                 path=gpu_lib.PATH_GATHER)
        assert plan["a_mode"] == amode, (shape.name, plan)
        x, w, b = workloads.make_inputs(shape)
        xd, wd, bd = x.to(dev), w.to(dev), b.to(dev)
        Ho = oracle.output_size(shape.H, shape.KH, shape.stride, shape.pad, shape.dilation)
        Wo = oracle.output_size(shape.W, shape.KW, shape.stride, shape.pad, shape.dilation)
        y = torch.full((shape.N, Ho, Wo, shape.C_out), float("nan"),
                       dtype=torch.float32 if f32 else torch.bfloat16, device=dev)
        assert noalloc(gpu_lib, xd, wd, bd, shape, y, f32) == 0
        st, code = gpu_lib.check_device_errors()
        assert st == 0, "device error word %#x" % code
        ref, mag = oracle.conv2d_direct(workloads.bits(x), workloads.bits(w), workloads.bits(b),
                                        shape.stride, shape.pad, shape.dilation)
        check(y.double().cpu().numpy(), ref, mag, shape.name)


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
    assert bool(torch.all(y3 == 0))  # a rejected call queues nothing
