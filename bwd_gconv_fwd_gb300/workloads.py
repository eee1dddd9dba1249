"""Seeded synthetic workloads for grouped 2D convolution.

This module only draws inputs: shapes, distributions, seeds and the one-time
rounding of fp32 draws to the storage dtype.  It holds none of the convolution
arithmetic, imports nothing else from this package, and is the one module that
both the CUDA path (through tests and the benchmark) and the fp64 oracle are fed
from, so both see bit-identical inputs.

Geometry tuples follow the C ABI order:
``(N, C_in, H, W, C_out, kH, kW, stride, pad_top, pad_bottom, pad_left, pad_right,
dilation, groups)``.

Workload recipe (each tensor drawn in fp32 with ``torch.Generator`` seeded
``seed + k``, k = 0 for x, 1 for w, 2 for bias, 3 for gradOutput, then rounded
once, round-to-nearest-even, to the storage dtype):

* ``tiny_g5``   -- the NNlib.jl grouped-conv timing example ("Support groups in
  DenseConvDims"): x [2,100,28,28] U[0,1), w [15,20,3,3] U[0,1), bias U[-1,1),
  gradOutput U[-1,1); groups 5, no padding; fp32 storage.
* ``alexnet_g2`` -- AlexNet-style 2-group layer (the caffe nets that motivated
  groups in clnn issue #4): x [128,96,27,27] N(0,1), w [256,48,5,5]
  N(0, sd=1/sqrt(1200)), bias N(0, sd=0.1), gradOutput N(0,1); pad 2; bf16.
* ``fc_mode``   -- input size == kernel size ("SpatialConvolution running in
  fully-connected mode is very slow"): x [1600,256,6,6] N(0,1),
  w [4096,256,6,6] N(0, sd=1/sqrt(9216)), bias N(0, sd=0.1), gradOutput N(0,1).
  Variants: ``fc_mode_ones_x`` (x = 1, gradOutput = 1) and ``fc_mode_all_ones``
  (the page's script: x, w, bias and gradOutput all 1).
* ``dense3x3``  -- x [32,64,56,56], w [64,64,3,3] N(0, sd=1/24), pad 1; and
  ``dense3x3_s2_asym`` with pads top/bottom/left/right 0/1/0/1, stride 2.
* ``resnext_g32`` -- x [64,128,56,56], w [128,4,3,3] N(0, sd=1/6), groups 32, pad 1;
  and ``depthwise`` x [64,256,56,56], w [256,1,3,3] N(0, sd=1/3), groups 256.
* ``model_zoo(N)`` -- a shape sweep: the grouped 3x3 layers of ResNeXt-50 (32x4d) and
  the depthwise 3x3 layers of MobileNet-v2 (stride 1 and 2, pad 1), batch N.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

SEED = 1234


@dataclass(frozen=True)
class Workload:
    name: str
    geom: tuple
    dtype: str                       # "bf16" or "f32": storage dtype of x, w, bias, gradOutput
    x: tuple = ("normal", 1.0)
    w: tuple = ("normal", 1.0)
    b: tuple = ("normal", 0.1)
    dy: tuple = ("normal", 1.0)
    note: str = ""
    extra: dict = field(default_factory=dict)


def _g(N, Cin, H, W, Cout, kH, kW, s=1, pt=0, pb=0, pl=0, pr=0, d=1, G=1):
    return (N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G)


WORKLOADS = {
    "tiny_g5": Workload("tiny_g5", _g(2, 100, 28, 28, 15, 3, 3, G=5), "f32",
                        x=("uniform", 0.0, 1.0), w=("uniform", 0.0, 1.0),
                        b=("uniform", -1.0, 1.0), dy=("uniform", -1.0, 1.0)),
    "alexnet_g2": Workload("alexnet_g2", _g(128, 96, 27, 27, 256, 5, 5, 1, 2, 2, 2, 2, 1, 2), "bf16",
                           w=("normal", 1.0 / math.sqrt(48 * 25))),
    "fc_mode": Workload("fc_mode", _g(1600, 256, 6, 6, 4096, 6, 6), "bf16",
                        w=("normal", 1.0 / math.sqrt(9216))),
    "fc_mode_ones_x": Workload("fc_mode_ones_x", _g(1600, 256, 6, 6, 4096, 6, 6), "bf16",
                               x=("const", 1.0), w=("normal", 1.0 / math.sqrt(9216)),
                               dy=("const", 1.0)),
    "fc_mode_all_ones": Workload("fc_mode_all_ones", _g(1600, 256, 6, 6, 4096, 6, 6), "bf16",
                                 x=("const", 1.0), w=("const", 1.0), b=("const", 1.0),
                                 dy=("const", 1.0)),
    "dense3x3": Workload("dense3x3", _g(32, 64, 56, 56, 64, 3, 3, 1, 1, 1, 1, 1), "bf16",
                         w=("normal", 1.0 / 24.0)),
    "dense3x3_s2_asym": Workload("dense3x3_s2_asym", _g(32, 64, 56, 56, 64, 3, 3, 2, 0, 1, 0, 1), "bf16",
                                 w=("normal", 1.0 / 24.0)),
    "resnext_g32": Workload("resnext_g32", _g(64, 128, 56, 56, 128, 3, 3, 1, 1, 1, 1, 1, 1, 32), "bf16",
                            w=("normal", 1.0 / 6.0)),
    "depthwise": Workload("depthwise", _g(64, 256, 56, 56, 256, 3, 3, 1, 1, 1, 1, 1, 1, 256), "bf16",
                          w=("normal", 1.0 / 3.0)),
}



def _zoo(name, N, C, HW, G, s):
    """A 3x3, pad-1 grouped or depthwise layer of a model-zoo network (C in = C out)."""
    return Workload(name, _g(N, C, HW, HW, C, 3, 3, s, 1, 1, 1, 1, 1, G), "bf16",
                    w=("normal", 1.0 / math.sqrt((C // G) * 9)))


def model_zoo(N):
    """Shape sweep of the grouped 3x3 layers of ResNeXt-50 (32x4d) and the depthwise 3x3
    layers of MobileNet-v2 at 224x224 input (the networks the pages validate grouped
    convolutions on), batch N; weights N(0, sd = 1/sqrt(fan_in)), everything else N(0, 1)
    or N(0, 0.1) for the bias, bf16 storage."""
    rx = [("resnext_s1_128x56", 128, 56, 1), ("resnext_s2_256x56", 256, 56, 2), ("resnext_s1_256x28", 256, 28, 1),
          ("resnext_s2_512x28", 512, 28, 2), ("resnext_s1_512x14", 512, 14, 1), ("resnext_s2_1024x14", 1024, 14, 2),
          ("resnext_s1_1024x7", 1024, 7, 1)]
    mb = [("mbv2_dw_32x112", 32, 112, 1), ("mbv2_dw_96x112_s2", 96, 112, 2), ("mbv2_dw_144x56", 144, 56, 1),
          ("mbv2_dw_144x56_s2", 144, 56, 2), ("mbv2_dw_192x28", 192, 28, 1), ("mbv2_dw_192x28_s2", 192, 28, 2),
          ("mbv2_dw_384x14", 384, 14, 1), ("mbv2_dw_576x14", 576, 14, 1), ("mbv2_dw_576x14_s2", 576, 14, 2),
          ("mbv2_dw_960x7", 960, 7, 1)]
    out = {nm: _zoo(nm, N, C, hw, 32, st) for nm, C, hw, st in rx}
    out.update({nm: _zoo(nm, N, C, hw, C, st) for nm, C, hw, st in mb})
    return out


def pointwise_zoo(N):
    """Shape sweep of 1x1 layers (stride 1, no padding): the channel-reducing and -expanding
    1x1 convolutions of ResNet-50 bottleneck blocks at 224x224 input, and a grouped 1x1
    layer, batch N; weights N(0, sd = 1/sqrt(fan_in)), bf16 storage."""
    layers = [("rn50_1x1_256to64_56", 256, 64, 56, 1), ("rn50_1x1_64to256_56", 64, 256, 56, 1),
              ("rn50_1x1_512to128_28", 512, 128, 28, 1), ("rn50_1x1_128to512_28", 128, 512, 28, 1),
              ("rn50_1x1_1024to256_14", 1024, 256, 14, 1), ("grouped_1x1_256to256_28_g4", 256, 256, 28, 4)]
    return {nm: Workload(nm, _g(N, ci, hw, hw, co, 1, 1, 1, 0, 0, 0, 0, 1, G), "bf16",
                         w=("normal", 1.0 / math.sqrt(ci // G)))
            for nm, ci, co, hw, G in layers}


def per_axis(geom):
    """The 16-integer form ``(N, C_in, H, W, C_out, kH, kW, stride_h, stride_w, pad_top,
    pad_bottom, pad_left, pad_right, dilation_h, dilation_w, groups)`` of a 14- or
    16-integer geometry (a 14-tuple has one stride and one dilation for both axes)."""
    geom = tuple(int(v) for v in geom)
    if len(geom) == 16:
        return geom
    N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G = geom
    return (N, Cin, H, W, Cout, kH, kW, s, s, pt, pb, pl, pr, d, d, G)


def out_hw(geom):
    """Output extent by the floor formula (shape bookkeeping for allocation only)."""
    N, Cin, H, W, Cout, kH, kW, sh, sw, pt, pb, pl, pr, dh, dw, G = per_axis(geom)
    ho = (H + pt + pb - dh * (kH - 1) - 1) // sh + 1
    wo = (W + pl + pr - dw * (kW - 1) - 1) // sw + 1
    return ho, wo


def tensor_shapes(geom):
    N, Cin, H, W, Cout, kH, kW, sh, sw, pt, pb, pl, pr, dh, dw, G = per_axis(geom)
    ho, wo = out_hw(geom)
    return dict(x=(N, Cin, H, W), w=(Cout, Cin // G, kH, kW), b=(Cout,), dy=(N, Cout, ho, wo))


def storage_dtype(dtype: str):
    return {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]


def draw(spec, shape, seed, dtype: str) -> torch.Tensor:
    """Draw one tensor on the CPU from its spec, then round once to the storage dtype."""
    gen = torch.Generator().manual_seed(int(seed))
    kind = spec[0]
    if kind == "normal":
        t = torch.randn(shape, generator=gen, dtype=torch.float32) * float(spec[1])
    elif kind == "uniform":
        lo, hi = float(spec[1]), float(spec[2])
        t = torch.rand(shape, generator=gen, dtype=torch.float32) * (hi - lo) + lo
    elif kind == "const":
        t = torch.full(shape, float(spec[1]), dtype=torch.float32)
    else:
        raise ValueError(f"unknown distribution {kind}")
    return t.to(storage_dtype(dtype)).contiguous()


def make_inputs(wl: Workload, seed: int = SEED, with_bias: bool = True):
    """x, w, bias (or None), gradOutput as CPU tensors in the storage dtype."""
    sh = tensor_shapes(wl.geom)
    x = draw(wl.x, sh["x"], seed + 0, wl.dtype)
    w = draw(wl.w, sh["w"], seed + 1, wl.dtype)
    b = draw(wl.b, sh["b"], seed + 2, wl.dtype) if with_bias else None
    dy = draw(wl.dy, sh["dy"], seed + 3, wl.dtype)
    return x, w, b, dy


def random_geometry(rng, max_n=2, max_c=24, max_hw=13, max_k=3, max_s=3, max_d=2, max_pad=2, axes=False):
    """A random small geometry that has at least one output pixel (parity sweeps); with
    axes=True a 16-integer geometry whose strides and dilations differ per axis."""
    if axes:
        while True:
            g14 = random_geometry(rng, max_n, max_c, max_hw, max_k, max_s, max_d, max_pad)
            N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G = g14
            sw = int(rng.integers(1, max_s + 1))
            dw = int(rng.integers(1, max_d + 1))
            geom = (N, Cin, H, W, Cout, kH, kW, s, sw, pt, pb, pl, pr, d, dw, G)
            ho, wo = out_hw(geom)
            if ho >= 1 and wo >= 1:
                return geom
    while True:
        G = int(rng.choice([1, 1, 2, 3, 4]))
        cgi = int(rng.integers(1, max(2, max_c // G) + 1))
        cgo = int(rng.integers(1, max(2, max_c // G) + 1))
        N = int(rng.integers(1, max_n + 1))
        H = int(rng.integers(1, max_hw + 1))
        W = int(rng.integers(1, max_hw + 1))
        kH = int(rng.integers(1, max_k + 1))
        kW = int(rng.integers(1, max_k + 1))
        s = int(rng.integers(1, max_s + 1))
        d = int(rng.integers(1, max_d + 1))
        pads = [int(v) for v in rng.integers(0, max_pad + 1, size=4)]
        geom = (N, cgi * G, H, W, cgo * G, kH, kW, s, *pads, d, G)
        ho, wo = out_hw(geom)
        if ho >= 1 and wo >= 1:
            return geom
