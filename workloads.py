"""Seeded synthetic convolution workloads.

The one module the GPU-side tests/benchmark and the CPU oracle both draw
inputs from.  It holds shapes and random-number recipes only: none of the
convolution's arithmetic lives here.

Recipe (every workload): one CPU ``torch.Generator`` seeded per workload
draws, in this order, x in logical [N][C_in][H][W], w in [C_out][C_in][KH][KW]
and bias in [C_out], each in fp32 from a normal distribution, then casts
them to bf16 and stores them channels-last (x as [N][H][W][C_in], w as
[C_out][KH][KW][C_in]).  x ~ N(0, 1); w ~ N(0, 1/(C_in*KH*KW)) (variance,
the fan-in scale); bias ~ N(0, 0.1^2) (standard deviation 0.1).  The tiny
case's w ~ N(0, 1/27) is the same rule at C_in*KH*KW = 27.
"""
from __future__ import annotations

from dataclasses import dataclass, field, asdict

import torch


@dataclass(frozen=True)
class ConvShape:
    name: str
    N: int
    C_in: int
    H: int
    W: int
    C_out: int
    KH: int
    KW: int
    stride: int = 1
    pad: int = 0
    dilation: int = 1
    out_f32: bool = False
    seed: int = 0
    bias: bool = True

    def as_dict(self):
        return asdict(self)

    def scaled(self, N: int, name_suffix: str = "") -> "ConvShape":
        d = asdict(self)
        d["N"] = N
        d["name"] = self.name + name_suffix
        return ConvShape(**d)


def _sweep():
    s = []
    j = 0

    def add(name, **kw):
        nonlocal j
        s.append(ConvShape(name=name, N=128, seed=2000 + j, **kw))
        j += 1

    add("sweep_3x3_64c_112", C_in=64, H=112, W=112, C_out=64, KH=3, KW=3, pad=1)
    add("sweep_3x3_128c_56", C_in=128, H=56, W=56, C_out=128, KH=3, KW=3, pad=1)
    add("sweep_3x3_256c_28", C_in=256, H=28, W=28, C_out=256, KH=3, KW=3, pad=1)
    add("sweep_3x3_512c_14", C_in=512, H=14, W=14, C_out=512, KH=3, KW=3, pad=1)
    add("sweep_3x3_512c_7", C_in=512, H=7, W=7, C_out=512, KH=3, KW=3, pad=1)
    add("sweep_3x3_d2_256c_28", C_in=256, H=28, W=28, C_out=256, KH=3, KW=3, pad=2, dilation=2)
    add("sweep_5x5_96to256_27", C_in=96, H=27, W=27, C_out=256, KH=5, KW=5, pad=2)
    add("sweep_1x1_512to2048_7", C_in=512, H=7, W=7, C_out=2048, KH=1, KW=1)
    add("sweep_3x3_s2_256to512_28", C_in=256, H=28, W=28, C_out=512, KH=3, KW=3, stride=2, pad=1)
    add("sweep_11x11_s4_3to64_224", C_in=3, H=224, W=224, C_out=64, KH=11, KW=11, stride=4, pad=2)
    add("sweep_fullspatial_7x7_512to4096", C_in=512, H=7, W=7, C_out=4096, KH=7, KW=7)
    add("sweep_3x3_32c_150", C_in=32, H=150, W=150, C_out=32, KH=3, KW=3, pad=1)
    return s


TINY = ConvShape("tiny_3to4_8x8_3x3", N=1, C_in=3, H=8, W=8, C_out=4, KH=3, KW=3,
                 stride=1, pad=1, out_f32=True, seed=1000)
RESNET_3X3 = ConvShape("resnet_3x3_64to128_56", N=32, C_in=64, H=56, W=56, C_out=128,
                       KH=3, KW=3, stride=1, pad=1, seed=1001)
POINTWISE_S1 = ConvShape("pointwise_1x1_256to64_56", N=32, C_in=256, H=56, W=56, C_out=64,
                         KH=1, KW=1, seed=1002)
POINTWISE_S2 = ConvShape("downsample_1x1_s2_256to512_56", N=32, C_in=256, H=56, W=56,
                         C_out=512, KH=1, KW=1, stride=2, seed=1102)
STEM_7X7 = ConvShape("stem_7x7_s2_3to64_224", N=64, C_in=3, H=224, W=224, C_out=64,
                     KH=7, KW=7, stride=2, pad=3, seed=1003)
STRIDED_3X3 = ConvShape("strided_3x3_s2_128to256_56", N=64, C_in=128, H=56, W=56,
                        C_out=256, KH=3, KW=3, stride=2, pad=1, seed=1103)
SWEEP = _sweep()

# The five workload groups, in order: the tiny parity case, the ResNet-style
# 3x3 layer (the headline benchmark), the two 1x1 layers, the two stem-era
# layers, and the 12-shape sweep at N=128.
GROUPS = {
    "tiny": [TINY],
    "resnet3x3": [RESNET_3X3],
    "pointwise": [POINTWISE_S1, POINTWISE_S2],
    "stem": [STEM_7X7, STRIDED_3X3],
    "sweep": SWEEP,
}
ALL = [c for g in GROUPS.values() for c in g]
BY_NAME = {c.name: c for c in ALL}


def make_inputs(shape: ConvShape, seed: int | None = None, device="cpu"):
    """(x, w, bias) as bf16 tensors: x [N,H,W,C_in], w [C_out,KH,KW,C_in], bias [C_out].

    bias is None when the shape has bias=False.  The draws come from a
    generator on `device` (the CPU by default, which the parity tests use; a
    CUDA generator gives the same distributions, not the same values).
    """
    g = torch.Generator(device=device).manual_seed(shape.seed if seed is None else seed)
    kw = dict(generator=g, dtype=torch.float32, device=device)
    x = torch.randn(shape.N, shape.C_in, shape.H, shape.W, **kw)
    w = torch.randn(shape.C_out, shape.C_in, shape.KH, shape.KW, **kw)
    w = w * (1.0 / (shape.C_in * shape.KH * shape.KW)) ** 0.5
    b = torch.randn(shape.C_out, **kw) * 0.1
    x = x.to(torch.bfloat16).permute(0, 2, 3, 1).contiguous()
    w = w.to(torch.bfloat16).permute(0, 2, 3, 1).contiguous()
    b = b.to(torch.bfloat16) if shape.bias else None
    return x, w, b


def bits(t: torch.Tensor):
    """numpy uint16 view of a CPU bf16 tensor's bit patterns."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")
