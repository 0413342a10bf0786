"""The oracle's pins have teeth: plant plausible slips in a copy of the C oracle.

Each mutant is a one-token edit of oracle/conv_oracle.c compiled into a
temporary library on the CPU.  The same comparison the pins make (against
torch's fp64 conv2d and the hand-worked golden example) must reject every
mutant, while the unmodified source passes it.  Geometries keep every
mutant's memory accesses inside its arrays.
"""
import ctypes
import json
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "conv_oracle.c")

MUTANTS = {
    "unmodified": (None, None),
    "bias_dropped": ("acc = bf16_to_double(bias[co]);", "acc = 0.0;"),
    "padding_sign": ("long h = ho * g->s + kh * g->d - g->p;",
                     "long h = ho * g->s + kh * g->d + g->p;"),
    "stride_dilation_swapped": ("long w = wo * g->s + kw * g->d - g->p;",
                                "long w = wo * g->d + kw * g->s - g->p;"),
    "kernel_transposed": ("wt[idx_w(g, co, ci, kh, kw)]", "wt[idx_w(g, co, ci, kw, kh)]"),
    "last_tap_dropped": ("for (long kw = 0; kw < g->KW; ++kw)",
                         "for (long kw = 0; kw + 1 < g->KW; ++kw)"),
    "output_size_off_by_one": ("return span / s + 1;", "return (span + 1) / s + 1;"),
}


def build_mutant(name, tmpdir):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    if old is not None:
        assert src.count(old) == 1, name
        src = src.replace(old, new)
    c = os.path.join(tmpdir, name + ".c")
    so = os.path.join(tmpdir, name + ".so")
    with open(c, "w") as f:
        f.write(src)
    subprocess.run(["gcc", "-O1", "-shared", "-fPIC", "-std=c99", c, "-o", so], check=True)
    lib = ctypes.CDLL(so)
    L, P = ctypes.c_long, ctypes.c_void_p
    lib.oracle_output_size.argtypes = [L] * 5
    lib.oracle_output_size.restype = L
    lib.oracle_conv2d_direct.argtypes = [P, P, P] + [L] * 10 + [P, P]
    lib.oracle_conv2d_direct.restype = ctypes.c_int
    return lib


def run(lib, x, w, b, s, p, d):
    xb, wb = workloads.bits(x), workloads.bits(w)
    bb = None if b is None else workloads.bits(b)
    N, H, W, C = xb.shape
    C_out, KH, KW, _ = wb.shape
    Ho = lib.oracle_output_size(H, KH, s, p, d)
    Wo = lib.oracle_output_size(W, KW, s, p, d)
    y = np.zeros((N, Ho, Wo, C_out))
    rc = lib.oracle_conv2d_direct(xb.ctypes.data, wb.ctypes.data,
                                  None if bb is None else bb.ctypes.data,
                                  N, C, H, W, C_out, KH, KW, s, p, d, y.ctypes.data, None)
    assert rc == 0
    return y


def pins_pass(lib):
    """The pin comparisons, reduced to one boolean."""
    cases = [(2, 3, 9, 9, 4, 3, 3, 2, 1, 2), (1, 4, 8, 7, 3, 3, 3, 1, 1, 1)]
    for (N, C, H, W, Co, KH, KW, s, p, d) in cases:
        shape = workloads.ConvShape("m", N=N, C_in=C, H=H, W=W, C_out=Co, KH=KH, KW=KW, seed=9)
        x, w, b = workloads.make_inputs(shape)
        y = run(lib, x, w, b, s, p, d)
        ref = F.conv2d(x.double().permute(0, 3, 1, 2), w.double().permute(0, 3, 1, 2),
                       b.double(), stride=s, padding=p, dilation=d).permute(0, 2, 3, 1).numpy()
        if y.shape != ref.shape or not np.allclose(y, ref, rtol=1e-12, atol=1e-12):
            return False
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "hand_conv_4x4.json")))
    x = torch.tensor(g["x_nchw"], dtype=torch.bfloat16).permute(0, 2, 3, 1).contiguous()
    w = torch.tensor(g["w_oihw"], dtype=torch.bfloat16).permute(0, 2, 3, 1).contiguous()
    b = torch.tensor(g["bias"], dtype=torch.bfloat16)
    for c in g["cases"]:
        y = run(lib, x, w, b, c["stride"], c["pad"], c["dilation"])
        expect = np.array(c["y_nchw"]).transpose(0, 2, 3, 1)
        if y.shape != expect.shape or not np.array_equal(y, expect):
            return False
    return True


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistakes(name):
    with tempfile.TemporaryDirectory() as d:
        lib = build_mutant(name, d)
        assert pins_pass(lib) == (name == "unmodified")
