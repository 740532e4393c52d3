"""Seeded synthetic inputs for the convolution workloads.

This module only describes workloads and draws their random inputs. It holds
none of the convolution's arithmetic (no output-size rule, no accumulation),
so the CUDA path and the CPU oracle can both be fed from it without sharing
any part of the method.

Workloads follow the envelope of the direct-stencil template described in
executorch PR #25085 ("Route 2-D depthwise and few-channel grouped
convolutions to a Triton direct-stencil kernel", description, second
paragraph): depthwise and grouped 2-D convolution with up to 8 input channels
per group, any channel multiplier, kernels up to 9x9, fp32/fp16/bf16, NCHW or
channels-last inputs, optional bias and asymmetric padding.

Recipe: values are drawn in fp32 from a CPU ``torch.Generator`` seeded with
``1000 * workload_id + {0: x, 1: w, 2: bias, 3: output gradient}``, cast to
the workload dtype and laid out in its memory format.  Weight variance is
``1 / fan_in`` with ``fan_in = Cin_g * KH * KW`` (Cin_g = C_in / groups, the
input channels one output sums over in the forward direction).  Where a bias
distribution is not stated it is U[-0.1, 0.1]; output gradients are N(0, 1).

Beyond that envelope, workloads may be dilated, 1-D (``spatial_dims = 1``:
x is [N, C, L], w [C_out, Cin_g, K], with H = KH = 1 in the description) or
transposed (w is [C_in, C_out / groups, KH, KW], the transposed convolution
of executorch PR #25091).
"""

from __future__ import annotations

import dataclasses
from typing import Optional, Tuple

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class ConvWorkload:
    """One convolution problem: shapes, geometry, dtype, layout and input law."""

    name: str
    wid: int                      # seed base: 1000 * wid
    N: int
    C_in: int
    H: int
    W: int
    C_out: int
    groups: int
    KH: int
    KW: int
    stride: Tuple[int, int]
    pad_before: Tuple[int, int]
    pad_after: Tuple[int, int]
    dtype: str                    # "f32" | "f16" | "bf16"
    channels_last: bool
    bias: bool
    x_law: str = "normal"         # "normal": N(0,1); "uniform": U[-1,1]
    b_lo: float = -0.1
    b_hi: float = 0.1
    dilation: Tuple[int, int] = (1, 1)
    transposed: bool = False
    output_padding: Tuple[int, int] = (0, 0)
    spatial_dims: int = 2         # 1: x [N, C, L] (H = KH = 1), channels_last = NLC

    @property
    def cin_g(self) -> int:
        return self.C_in // self.groups

    @property
    def fan_in(self) -> int:
        return self.cin_g * self.KH * self.KW

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    def replace(self, **kw) -> "ConvWorkload":
        return dataclasses.replace(self, **kw)


# The five benchmark workloads (a depthwise fp32 NCHW case, a MobileNetV2-style
# bf16 channels-last depthwise layer at stride 1 and 2, a large-kernel 7x7
# depthwise layer, a multiplier-4 fp16 NCHW layer with 'same' asymmetric
# padding, and a few-channel grouped 9x9 stride-2 layer), then the workloads
# of the wider envelope: the MobileNetV2 layer with dilation 2 (as in
# atrous / dilated backbones), a causal depthwise 1-D convolution of kernel 4
# over long channels-last sequences (the short convolution of state-space
# sequence models: padding 3 before, 0 after), and a depthwise transposed
# 1-D upsampling of kernel 4, stride 2 (the shape executorch PR #25091's
# benchmark adds).
WORKLOADS = {
    "dw3x3_f32_nchw": ConvWorkload(
        "dw3x3_f32_nchw", 1, N=1, C_in=32, H=56, W=56, C_out=32, groups=32,
        KH=3, KW=3, stride=(1, 1), pad_before=(1, 1), pad_after=(1, 1),
        dtype="f32", channels_last=False, bias=True, x_law="uniform"),
    "mbv2_dw3x3_s1_bf16_cl": ConvWorkload(
        "mbv2_dw3x3_s1_bf16_cl", 2, N=32, C_in=144, H=56, W=56, C_out=144,
        groups=144, KH=3, KW=3, stride=(1, 1), pad_before=(1, 1),
        pad_after=(1, 1), dtype="bf16", channels_last=True, bias=True),
    "mbv2_dw3x3_s2_bf16_cl": ConvWorkload(
        "mbv2_dw3x3_s2_bf16_cl", 2, N=32, C_in=144, H=56, W=56, C_out=144,
        groups=144, KH=3, KW=3, stride=(2, 2), pad_before=(1, 1),
        pad_after=(1, 1), dtype="bf16", channels_last=True, bias=True),
    "dw7x7_bf16_cl": ConvWorkload(
        "dw7x7_bf16_cl", 3, N=128, C_in=96, H=56, W=56, C_out=96, groups=96,
        KH=7, KW=7, stride=(1, 1), pad_before=(3, 3), pad_after=(3, 3),
        dtype="bf16", channels_last=True, bias=True),
    "dw4x4_m4_f16_nchw": ConvWorkload(
        "dw4x4_m4_f16_nchw", 4, N=16, C_in=64, H=112, W=112, C_out=256,
        groups=64, KH=4, KW=4, stride=(1, 1), pad_before=(1, 1),
        pad_after=(2, 2), dtype="f16", channels_last=False, bias=False,
        x_law="uniform"),
    "grp4x8_9x9_s2_bf16_cl": ConvWorkload(
        "grp4x8_9x9_s2_bf16_cl", 5, N=8, C_in=256, H=128, W=128, C_out=512,
        groups=64, KH=9, KW=9, stride=(2, 2), pad_before=(4, 4),
        pad_after=(4, 4), dtype="bf16", channels_last=True, bias=True),
    "mbv2_dw3x3_d2_bf16_cl": ConvWorkload(
        "mbv2_dw3x3_d2_bf16_cl", 6, N=32, C_in=144, H=56, W=56, C_out=144,
        groups=144, KH=3, KW=3, stride=(1, 1), pad_before=(2, 2),
        pad_after=(2, 2), dtype="bf16", channels_last=True, bias=True, dilation=(2, 2)),
    "causal_dw1d_k4_bf16_nlc": ConvWorkload(
        "causal_dw1d_k4_bf16_nlc", 7, N=8, C_in=2048, H=1, W=4096, C_out=2048,
        groups=2048, KH=1, KW=4, stride=(1, 1), pad_before=(0, 3), pad_after=(0, 0),
        dtype="bf16", channels_last=True, bias=True, spatial_dims=1),
    "upsample_dwT1d_k4s2_bf16_nlc": ConvWorkload(
        "upsample_dwT1d_k4s2_bf16_nlc", 8, N=8, C_in=512, H=1, W=8192, C_out=512,
        groups=512, KH=1, KW=4, stride=(1, 2), pad_before=(0, 1), pad_after=(0, 1),
        dtype="bf16", channels_last=True, bias=True, spatial_dims=1, transposed=True),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def make_inputs(wl: ConvWorkload, device: str | torch.device = "cpu",
                seed_base: Optional[int] = None):
    """Draw (x, w, bias) for a workload.

    ``x`` has logical shape [N, C_in, H, W] and is laid out channels-last when
    the workload says so; ``w`` is a dense [C_out, C_in/groups, KH, KW] tensor
    ([C_in, C_out/groups, KH, KW] when transposed); ``bias`` is a dense
    [C_out] tensor or None.  All share the workload dtype.  1-D workloads
    drop the height dims: x [N, C_in, L] (channels-last = NLC order) and w
    [.., .., K].
    """
    base = 1000 * wl.wid if seed_base is None else seed_base
    dt = wl.torch_dtype
    shape_x = (wl.N, wl.C_in, wl.H, wl.W)
    if wl.x_law == "uniform":
        x = torch.rand(shape_x, generator=_gen(base + 0), dtype=torch.float32) * 2.0 - 1.0
    elif wl.x_law == "normal":
        x = torch.randn(shape_x, generator=_gen(base + 0), dtype=torch.float32)
    else:
        raise ValueError(f"unknown x law {wl.x_law!r}")
    w_shape = ((wl.C_in, wl.C_out // wl.groups, wl.KH, wl.KW) if wl.transposed
               else (wl.C_out, wl.cin_g, wl.KH, wl.KW))
    w = torch.randn(w_shape, generator=_gen(base + 1),
                    dtype=torch.float32) * (1.0 / wl.fan_in) ** 0.5
    b = None
    if wl.bias:
        b = torch.rand((wl.C_out,), generator=_gen(base + 2), dtype=torch.float32)
        b = b * (wl.b_hi - wl.b_lo) + wl.b_lo
    x = x.to(dt)
    if wl.spatial_dims == 1:
        x = x[:, :, 0, :]
        w = w[:, :, 0, :]
        if wl.channels_last:
            x = x.permute(0, 2, 1).contiguous().permute(0, 2, 1)
    elif wl.channels_last:
        x = x.contiguous(memory_format=torch.channels_last)
    w = w.to(dt)
    b = b.to(dt) if b is not None else None
    if str(device) != "cpu":
        x = x.to(device)
        w = w.to(device)
        b = b.to(device) if b is not None else None
    return x, w, b


def small_variant(wl: ConvWorkload, N: int = 1, H: Optional[int] = None,
                  W: Optional[int] = None, C_div: int = 1) -> ConvWorkload:
    """A reduced copy of a workload (fewer images, smaller planes or fewer
    groups) with the same dtype, layout, kernel, stride, padding and group
    shape, for cases the oracle must finish in seconds."""
    G = max(1, wl.groups // C_div)
    return wl.replace(name=wl.name + "_small", N=N,
                      H=H if H is not None else wl.H,
                      W=W if W is not None else wl.W,
                      C_in=wl.cin_g * G, C_out=(wl.C_out // wl.groups) * G,
                      groups=G)


def make_grad(wl: ConvWorkload, out_shape, device: str | torch.device = "cpu"):
    """Draw an output gradient gy ~ N(0, 1) of the given logical shape
    (the caller supplies the output size), laid out like the workload's x."""
    g = torch.randn(tuple(out_shape), generator=_gen(1000 * wl.wid + 3), dtype=torch.float32)
    g = g.to(wl.torch_dtype)
    if wl.channels_last:
        if g.dim() == 4:
            g = g.contiguous(memory_format=torch.channels_last)
        elif g.dim() == 3:
            g = g.permute(0, 2, 1).contiguous().permute(0, 2, 1)
    return g.to(device) if str(device) != "cpu" else g
