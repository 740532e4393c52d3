"""Timed schedule choice (executorch PR #25085, description, second
paragraph: the direct-stencil template's schedules are timed and the fastest
kept): conv_autotune times every schedule that takes a call, records the
fastest for the call's shape, and later AUTO calls of that shape run it; the
result stays within the parity tolerance of the fp64 oracle."""

import ctypes

import pytest
import torch

import grouped_convolution_gb300 as gc
import oracle
from grouped_convolution_gb300.inputs import WORKLOADS, make_inputs, small_variant


def _check(wl, x, w, b, y):
    ref, bound = oracle.reference(wl, x.cpu(), w.cpu(), None if b is None else b.cpu())
    assert tuple(y.shape) == ref.shape
    bad = oracle.violations(y.cpu(), ref, bound, wl.dtype)
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} outside tolerance"


@pytest.mark.gpu
@pytest.mark.parametrize("name,red", [
    ("mbv2_dw3x3_s1_bf16_cl", dict(N=4)),
    ("dw4x4_m4_f16_nchw", dict(N=1, H=40, W=40)),
    ("upsample_dwT1d_k4s2_bf16_nlc", dict(N=2, W=2000)),
])
def test_autotune_records_the_fastest(name, red):
    gc.build()
    wl = small_variant(WORKLOADS[name], **red)
    x, w, b = make_inputs(wl, device="cuda")
    gc.conv_autotune_clear()
    d = gc.bind(x, w, b, wl.stride, wl.pad_before, wl.pad_after, wl.dilation, wl.groups,
                wl.transposed, wl.output_padding)
    y = gc.empty_output(d, x)
    heuristic = gc.conv_select_schedule(d, x, w, b, y)
    best, us = gc.conv_autotune(d, x, w, b, y, reps=3)
    torch.cuda.synchronize()
    assert us > 0 and best in gc.SCHEDULES
    _check(wl, x, w, b, y)                       # y holds the chosen schedule's result
    assert gc.conv_select_schedule(d, x, w, b, y) == best
    y2 = gc.empty_output(d, x)
    gc.run(d, x, w, b, y2)
    torch.cuda.synchronize()
    _check(wl, x, w, b, y2)
    # an explicit schedule on the desc is not overridden by the record
    d.schedule = gc.SCHEDULES["dw_flat"]
    assert gc.conv_select_schedule(d, x, w, b, y) == "dw_flat"
    d.schedule = -1
    gc.conv_autotune_clear()
    assert gc.conv_select_schedule(d, x, w, b, y) == heuristic


def test_autotune_argument_errors():
    gc.build()
    lib = gc._load()
    d = gc.conv_bind(((1, 16, 8, 8), (1024, 1, 128, 16)), ((16, 1, 3, 3), (9, 9, 3, 1)),
                     None, 1, 1, 1, 1, 16, dtype="bfloat16")
    fake = 1 << 20
    out = ctypes.c_int32()
    assert lib.conv_autotune(ctypes.byref(d), fake, fake, None, fake, None, 0,
                             ctypes.byref(out), None) == 4          # reps < 1
    assert lib.conv_autotune(None, fake, fake, None, fake, None, 3, None, None) == 1
