"""Pins of the CPU oracle against things other than itself.

Each test fixes the oracle to an independent source: torch's CPU conv2d and
unfold (library routines) in fp64, the GEMM the tutorial lowers to, closed
forms (delta kernels, all-ones inputs), the invariants the pages state, and a
hand-worked example stored under tests/golden/.  The cases are chosen so that
a plausible slip (dropped bias, padding sign, kh/kw or H/W swapped, dilation
applied to the wrong term, stride misplaced) fails at least one of them.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_case(seed, N, C_in, H, W, C_out, KH, KW, with_bias=True):
    shape = workloads.ConvShape("t", N=N, C_in=C_in, H=H, W=W, C_out=C_out, KH=KH, KW=KW,
                                seed=seed, bias=with_bias)
    return workloads.make_inputs(shape)


def torch_ref(x, w, b, s, p, d):
    """torch.nn.functional.conv2d in fp64 on NCHW views, returned NHWC."""
    xd = x.double().permute(0, 3, 1, 2)
    wd = w.double().permute(0, 3, 1, 2)
    bd = None if b is None else b.double()
    return F.conv2d(xd, wd, bd, stride=s, padding=p, dilation=d).permute(0, 2, 3, 1).numpy()


GEOMS = [
    # N, C_in, H, W, C_out, KH, KW, s, p, d
    (1, 3, 8, 8, 4, 3, 3, 1, 1, 1),
    (2, 5, 9, 7, 3, 3, 2, 1, 0, 1),   # KH != KW, H != W
    (2, 4, 11, 10, 6, 3, 3, 2, 1, 1),  # stride 2, odd size
    (1, 6, 12, 13, 5, 3, 3, 1, 2, 2),  # dilation 2
    (2, 3, 15, 14, 4, 5, 3, 3, 2, 2),  # everything at once
    (1, 8, 7, 7, 7, 1, 1, 1, 0, 1),    # 1x1
    (2, 8, 8, 8, 4, 1, 1, 2, 0, 1),    # 1x1 stride 2
    (1, 2, 6, 5, 3, 6, 5, 1, 0, 1),    # kernel covers the whole image
    (3, 2, 5, 5, 2, 2, 4, 3, 3, 1),    # pad larger than kernel overlap
]


@pytest.mark.parametrize("geom", GEOMS)
@pytest.mark.parametrize("with_bias", [True, False])
def test_direct_matches_torch_conv2d_fp64(geom, with_bias):
    N, C_in, H, W, C_out, KH, KW, s, p, d = geom
    x, w, b = rand_case(7 + sum(geom), N, C_in, H, W, C_out, KH, KW, with_bias)
    y, mag = oracle.conv2d_direct(workloads.bits(x), workloads.bits(w),
                                  None if b is None else workloads.bits(b), s, p, d)
    ref = torch_ref(x, w, b, s, p, d)
    assert y.shape == ref.shape
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    assert np.all(mag >= np.abs(y) - 1e-12)


@pytest.mark.parametrize("geom", GEOMS)
def test_direct_matches_im2col_gemm(geom):
    """The tutorial's second route: im2col, then Y_col = X_col W_row^T, then bias."""
    N, C_in, H, W, C_out, KH, KW, s, p, d = geom
    x, w, b = rand_case(100 + sum(geom), N, C_in, H, W, C_out, KH, KW)
    xb, wb, bb = workloads.bits(x), workloads.bits(w), workloads.bits(b)
    y, _ = oracle.conv2d_direct(xb, wb, bb, s, p, d)
    y2 = oracle.conv2d_im2col_gemm(xb, wb, bb, s, p, d)
    np.testing.assert_allclose(y, y2, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("L,K,s,p,d", [
    (56, 3, 1, 1, 1), (224, 7, 2, 3, 1), (224, 11, 4, 2, 1), (28, 3, 1, 2, 2),
    (7, 7, 1, 0, 1), (27, 5, 1, 2, 1), (56, 1, 2, 0, 1), (150, 3, 1, 1, 1),
    (5, 3, 1, 0, 2), (10, 4, 3, 1, 2), (1, 1, 1, 0, 1), (9, 2, 5, 0, 3),
])
def test_output_size_matches_torch(L, K, s, p, d):
    got = oracle.output_size(L, K, s, p, d)
    xx = torch.zeros(1, 1, L, 1, dtype=torch.float64)
    ww = torch.zeros(1, 1, K, 1, dtype=torch.float64)
    ref = F.conv2d(xx, ww, stride=(s, 1), padding=(p, 0), dilation=(d, 1)).shape[2]
    assert got == ref
    if d == 1:  # the tutorial's printed form, section 5
        assert got == (L + 2 * p - K) // s + 1


def test_output_size_rejects_kernel_larger_than_padded_input():
    assert oracle.output_size(3, 5, 1, 0, 1) == 0
    assert oracle.output_size(5, 3, 1, 0, 3) == 0  # dilated extent 7 > 5
    x = np.zeros((1, 3, 3, 1), np.uint16)
    w = np.zeros((1, 5, 5, 1), np.uint16)
    with pytest.raises(ValueError):
        oracle.conv2d_direct(x, w, None, 1, 0, 1)


def test_pointwise_stride1_is_a_gemm():
    """1x1 stride-1 convolution is a plain GEMM over the channel axis."""
    x, w, b = rand_case(3, 2, 16, 5, 6, 9, 1, 1)
    xb, wb, bb = workloads.bits(x), workloads.bits(w), workloads.bits(b)
    y, _ = oracle.conv2d_direct(xb, wb, bb, 1, 0, 1)
    X = oracle.bf16_bits_to_f64(xb).reshape(-1, 16)
    Wm = oracle.bf16_bits_to_f64(wb).reshape(9, 16)
    ref = X @ Wm.T + oracle.bf16_bits_to_f64(bb)[None, :]
    np.testing.assert_allclose(y.reshape(-1, 9), ref, rtol=1e-12, atol=1e-12)


def test_full_spatial_kernel_is_a_dense_layer():
    """A kernel covering the whole H x W gives a 1x1 output equal to an FC layer
    on the flattened image ("Unifying Convolutions and GEMM", section 4)."""
    N, C, H, W, C_out = 3, 4, 5, 6, 7
    x, w, b = rand_case(11, N, C, H, W, C_out, H, W)
    xb, wb, bb = workloads.bits(x), workloads.bits(w), workloads.bits(b)
    y, _ = oracle.conv2d_direct(xb, wb, bb, 1, 0, 1)
    assert y.shape == (N, 1, 1, C_out)
    # flatten in logical (C, H, W) order on both sides, as the page does
    xf = x.double().permute(0, 3, 1, 2).reshape(N, -1).numpy()
    Wd = w.double().permute(0, 3, 1, 2).reshape(C_out, -1).numpy()
    ref = xf @ Wd.T + b.double().numpy()[None, :]
    np.testing.assert_allclose(y.reshape(N, C_out), ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("kh0,kw0,s,p,d", [(0, 0, 1, 1, 1), (2, 1, 1, 1, 1), (1, 2, 2, 2, 1),
                                            (2, 0, 1, 2, 2), (0, 2, 3, 1, 1)])
def test_delta_kernel_shifts_the_input(kh0, kw0, s, p, d):
    """w = delta at one tap and one channel: y[n,ho,wo,co] = x[n, ho*s+kh0*d-p, wo*s+kw0*d-p, ci0]
    (0 in the padding); closed form of the definition."""
    N, C, H, W, KH, KW, C_out = 2, 3, 7, 8, 3, 3, 2
    x, _, _ = rand_case(5, N, C, H, W, C_out, KH, KW)
    xf = x.double().numpy()
    w = torch.zeros(C_out, KH, KW, C, dtype=torch.bfloat16)
    ci_of = [1, 2]
    for co in range(C_out):
        w[co, kh0, kw0, ci_of[co]] = 1.0
    y, _ = oracle.conv2d_direct(workloads.bits(x), workloads.bits(w), None, s, p, d)
    H_out, W_out = y.shape[1], y.shape[2]
    for n, ho, wo, co in itertools.product(range(N), range(H_out), range(W_out), range(C_out)):
        h, ww = ho * s + kh0 * d - p, wo * s + kw0 * d - p
        ref = xf[n, h, ww, ci_of[co]] if (0 <= h < H and 0 <= ww < W) else 0.0
        assert y[n, ho, wo, co] == ref


@pytest.mark.parametrize("s,p,d", [(1, 1, 1), (2, 3, 1), (1, 2, 2), (3, 0, 1)])
def test_all_ones_counts_in_range_taps(s, p, d):
    """x = 1, w = 1, bias = b0: y = b0 + C_in * (#kh in range) * (#kw in range)."""
    N, C, H, W, KH, KW, C_out = 1, 5, 9, 6, 3, 4, 2
    one = 0x3F80  # bf16 bits of 1.0
    x = np.full((N, H, W, C), one, np.uint16)
    w = np.full((C_out, KH, KW, C), one, np.uint16)
    b = np.full((C_out,), 0x4000, np.uint16)  # 2.0
    y, mag = oracle.conv2d_direct(x, w, b, s, p, d)
    for ho in range(y.shape[1]):
        nh = sum(0 <= ho * s + kh * d - p < H for kh in range(KH))
        for wo in range(y.shape[2]):
            nw = sum(0 <= wo * s + kw * d - p < W for kw in range(KW))
            assert np.all(y[0, ho, wo, :] == 2.0 + C * nh * nw)
            assert np.all(mag[0, ho, wo, :] == 2.0 + C * nh * nw)


def test_hand_worked_golden_example():
    """A 4x4 image and a 3x3 kernel worked by hand (tests/golden/hand_conv_4x4.json)."""
    with open(os.path.join(GOLDEN, "hand_conv_4x4.json")) as f:
        g = json.load(f)
    x = torch.tensor(g["x_nchw"], dtype=torch.bfloat16).permute(0, 2, 3, 1).contiguous()
    w = torch.tensor(g["w_oihw"], dtype=torch.bfloat16).permute(0, 2, 3, 1).contiguous()
    b = torch.tensor(g["bias"], dtype=torch.bfloat16)
    for case in g["cases"]:
        y, _ = oracle.conv2d_direct(workloads.bits(x), workloads.bits(w), workloads.bits(b),
                                    case["stride"], case["pad"], case["dilation"])
        expect = np.array(case["y_nchw"], np.float64).transpose(0, 2, 3, 1)
        np.testing.assert_array_equal(y, expect)


def test_points_match_full_tensor():
    x, w, b = rand_case(21, 2, 6, 10, 9, 5, 3, 3)
    xb, wb, bb = workloads.bits(x), workloads.bits(w), workloads.bits(b)
    y, mag = oracle.conv2d_direct(xb, wb, bb, 2, 1, 1)
    rng = np.random.default_rng(0)
    pts = np.stack([rng.integers(0, y.shape[0], 40), rng.integers(0, y.shape[3], 40),
                    rng.integers(0, y.shape[1], 40), rng.integers(0, y.shape[2], 40)], 1)
    v, m = oracle.conv2d_points(xb, wb, bb, 2, 1, 1, pts)
    for i, (n, co, ho, wo) in enumerate(pts):
        assert v[i] == y[n, ho, wo, co]
        assert m[i] == mag[n, ho, wo, co]
    with pytest.raises(ValueError):
        oracle.conv2d_points(xb, wb, bb, 2, 1, 1, [[0, 0, 99, 0]])


def unfold_rows(x, KH, KW, s, p, d):
    """torch's own im2col (F.unfold), rows = output pixels, columns in (kh, kw, ci) order."""
    xd = x.double().permute(0, 3, 1, 2)
    N, C = xd.shape[:2]
    u = F.unfold(xd, (KH, KW), dilation=d, padding=p, stride=s)  # [N, C*KH*KW, L]
    u = u.reshape(N, C, KH, KW, -1).permute(0, 4, 2, 3, 1)      # [N, L, KH, KW, C]
    return u.reshape(-1, KH * KW * C).numpy()


@pytest.mark.parametrize("geom", GEOMS)
def test_im2col_matches_torch_unfold(geom):
    N, C_in, H, W, C_out, KH, KW, s, p, d = geom
    x, _, _ = rand_case(31, N, C_in, H, W, C_out, KH, KW)
    mine = oracle.im2col(oracle.bf16_bits_to_f64(workloads.bits(x)), KH, KW, s, p, d)
    np.testing.assert_array_equal(mine, unfold_rows(x, KH, KW, s, p, d))
    assert mine.size == oracle.im2col_elements(N, C_in, H, W, KH, KW, s, p, d)


@pytest.mark.parametrize("geom", GEOMS)
def test_indirection_buffer_reproduces_unfold(geom):
    """Gathering pixel vectors through the buffer (-1 -> zeros) rebuilds im2col."""
    N, C_in, H, W, C_out, KH, KW, s, p, d = geom
    x, _, _ = rand_case(41, N, C_in, H, W, C_out, KH, KW)
    buf = oracle.indirection_buffer(H, W, C_in, KH, KW, s, p, d)
    H_out = oracle.output_size(H, KH, s, p, d)
    W_out = oracle.output_size(W, KW, s, p, d)
    assert buf.shape == (H_out * W_out, KH * KW) and buf.dtype == np.int32
    flat = oracle.bf16_bits_to_f64(workloads.bits(x)).reshape(N, -1)
    rows = np.zeros((N, H_out * W_out, KH * KW, C_in))
    for pix in range(H_out * W_out):
        for t in range(KH * KW):
            o = buf[pix, t]
            assert o == -1 or (o % C_in == 0 and 0 <= o < H * W * C_in)
            if o >= 0:
                rows[:, pix, t, :] = flat[:, o:o + C_in]
    np.testing.assert_array_equal(rows.reshape(-1, KH * KW * C_in),
                                  unfold_rows(x, KH, KW, s, p, d))


@pytest.mark.parametrize("geom", GEOMS)
def test_im2win_windows_reproduce_unfold(geom):
    """Each output pixel's window in Win, read in (kw, kh, ci) order with taps d
    columns apart, is that pixel's im2col row (reordered from (kh, kw, ci))."""
    N, C_in, H, W, C_out, KH, KW, s, p, d = geom
    x, _, _ = rand_case(51, N, C_in, H, W, C_out, KH, KW)
    win = oracle.im2win(workloads.bits(x), KH, KW, s, p, d)
    H_out = oracle.output_size(H, KH, s, p, d)
    W_out = oracle.output_size(W, KW, s, p, d)
    W_used = (W_out - 1) * s + (KW - 1) * d + 1
    assert win.shape == (N, H_out, W_used, KH, C_in)
    assert win.size == oracle.im2win_elements(N, C_in, H, W, KH, KW, s, p, d)
    wf = oracle.bf16_bits_to_f64(win)
    rows = np.empty((N, H_out, W_out, KH, KW, C_in))
    for wo in range(W_out):
        for kw in range(KW):
            rows[:, :, wo, :, kw, :] = wf[:, :, wo * s + kw * d, :, :]
    np.testing.assert_array_equal(rows.reshape(-1, KH * KW * C_in),
                                  unfold_rows(x, KH, KW, s, p, d))
    if d == 1 and s == 1:
        # stride-1, undilated: one pixel's whole window is one contiguous run
        flat = win.reshape(N, H_out, -1)
        run = KW * KH * C_in
        for wo in range(W_out):
            seg = flat[:, :, wo * KH * C_in: wo * KH * C_in + run]
            assert seg.shape[-1] == run


def test_im2win_is_smaller_than_im2col_for_3x3():
    """The window-order buffer stores each input row once per output row instead of
    once per tap column: for KW > stride it is smaller than im2col."""
    args = (32, 64, 56, 56, 3, 3, 1, 1, 1)
    assert oracle.im2win_elements(*args) < oracle.im2col_elements(*args)


@pytest.mark.parametrize("geom", GEOMS)
def test_im2win_width_is_the_tightest_span_of_the_columns_read(geom):
    """The window-order buffer keeps one contiguous span of input columns per
    output row (the reading of the layout).  That span must contain every column
    the 7-loop convolution's index map reads (w = wo*s + kw*d - p) and start and
    end on a column that is read: no dead column at either end (a W_used that is
    too large would still reproduce unfold above) and none missing.  With
    stride > dilation the columns between read ones stay in the span.  The set
    of columns read is enumerated from the loop indices, not from the W_used
    formula."""
    N, C_in, H, W, C_out, KH, KW, s, p, d = geom
    x, _, _ = rand_case(52, N, C_in, H, W, C_out, KH, KW)
    win = oracle.im2win(workloads.bits(x), KH, KW, s, p, d)
    W_out = oracle.output_size(W, KW, s, p, d)
    read = {wo * s + kw * d - p for wo in range(W_out) for kw in range(KW)}
    # buffer column wc holds input column wc - p
    kept = [wc - p for wc in range(win.shape[2])]
    assert read <= set(kept)
    assert kept[0] == min(read) and kept[-1] == max(read)
    assert oracle.im2win_elements(N, C_in, H, W, KH, KW, s, p, d) == \
        N * win.shape[1] * (max(read) - min(read) + 1) * KH * C_in
