"""conv_backward_weight_noalloc, the weight / bias gradient for callers that
cannot allocate device memory (code inside a host framework that owns every
device allocation, or on a fixed memory budget): it takes no workspace and
uses the library's fixed device scratch buffer instead.

Checked through the C ABI against conv_backward_weight (the entry point with
a caller workspace) on the same inputs, within the parity tolerance the other
tests use, on two calls in a row (the second one finds the first one's
contents in the shared buffer), and against the fp64 oracle.  This file is
collected last so that a run stopping at the first failure has already run
every other test; it passes on its own in a fresh process too.
"""

import ctypes

import numpy as np
import pytest
import torch

import grouped_convolution_gb300 as gc
import oracle
from grouped_convolution_gb300.inputs import WORKLOADS, make_grad, make_inputs, small_variant

pytestmark = pytest.mark.gpu

CASES = [
    # workload, reduced copy: (N, H, W) -- channels-last depthwise (registers
    # form of the partial pass) and a grouped / NCHW one (generic form)
    ("mbv2_dw3x3_s1_bf16_cl", (4, 28, 30)),
    ("mbv2_dw3x3_s2_bf16_cl", (4, 28, 30)),
    ("dw4x4_m4_f16_nchw", (2, 20, 21)),
    ("grp4x8_9x9_s2_bf16_cl", (1, 24, 26)),
]


def _call_noalloc(lib, d, x, gy, dw, db):
    return lib.conv_backward_weight_noalloc(ctypes.byref(d), x.data_ptr(), gy.data_ptr(),
                                            dw.data_ptr(), db.data_ptr(),
                                            torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name,red", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_workspace_entry_point(name, red):
    gc.build()
    lib = gc._load()
    N, H, W = red
    wl = small_variant(WORKLOADS[name], N=N, H=H, W=W, C_div=4 if "grp" in name else 1)
    x, w, _ = make_inputs(wl)
    d = gc.conv_bind(x, w, None, wl.stride, wl.pad_before, wl.pad_after, 1, wl.groups)
    ysz, _ = gc.out_shape_and_stride(d)
    gy = make_grad(wl, ysz)
    dev = torch.device("cuda")
    xd, gyd = x.to(dev), gy.to(dev)
    assert gc.conv_backward_weight_workspace_size(d) <= gc.conv_backward_weight_noalloc_limit()

    # the entry point with a caller workspace
    ref_dw = torch.empty(tuple(w.shape), dtype=w.dtype, device=dev)
    ref_db = torch.empty(d.C_out, dtype=w.dtype, device=dev)
    nbytes = gc.conv_backward_weight_workspace_size(d)
    ws = torch.empty(nbytes // 4 + 4, dtype=torch.float32, device=dev)
    gc.conv_backward_weight(d, xd, gyd, ref_dw, ref_db, ws, nbytes)

    g = oracle.conv2d_backward(x, w, gy, wl.stride, wl.pad_before, wl.pad_after, wl.groups,
                               need=("dw", "db"))
    for call in range(2):
        dw = torch.full(tuple(w.shape), float("nan"), dtype=w.dtype, device=dev)
        db = torch.full((d.C_out,), float("nan"), dtype=w.dtype, device=dev)
        assert _call_noalloc(lib, d, xd, gyd, dw, db) == 0, f"call {call}"
        torch.cuda.synchronize()
        # same kernels, same order: the same bits as the workspace entry point
        assert torch.equal(dw, ref_dw), f"call {call}: dw differs"
        assert torch.equal(db, ref_db), f"call {call}: db differs"
        # and within the parity tolerance of the fp64 oracle
        for got, (ref, bound) in ((dw, g["dw"]), (db, g["db"])):
            assert not oracle.violations(got.cpu(), ref, bound, wl.dtype).any(), f"call {call}"


def _problem(name, N, H, W):
    wl = small_variant(WORKLOADS[name], N=N, H=H, W=W)
    x, w, _ = make_inputs(wl)
    d = gc.conv_bind(x, w, None, wl.stride, wl.pad_before, wl.pad_after, 1, wl.groups)
    ysz, _ = gc.out_shape_and_stride(d)
    gy = make_grad(wl, ysz)
    dev = torch.device("cuda")
    return wl, d, w, x.to(dev), gy.to(dev)


def test_noalloc_small_call_after_large_one():
    # The shared buffer keeps what the larger call left there; the smaller
    # call must not read any of it: bit-equal to the workspace entry point.
    gc.build()
    lib = gc._load()
    dev = torch.device("cuda")
    big = _problem("mbv2_dw3x3_s2_bf16_cl", 16, 56, 56)
    small = _problem("mbv2_dw3x3_s1_bf16_cl", 1, 9, 11)
    limit = gc.conv_backward_weight_noalloc_limit()
    assert (gc.conv_backward_weight_workspace_size(small[1])
            < gc.conv_backward_weight_workspace_size(big[1]) <= limit)
    for wl, d, w, xd, gyd in (big, small):
        dw = torch.empty(tuple(w.shape), dtype=w.dtype, device=dev)
        db = torch.empty(d.C_out, dtype=w.dtype, device=dev)
        assert _call_noalloc(lib, d, xd, gyd, dw, db) == 0
        nbytes = gc.conv_backward_weight_workspace_size(d)
        ws = torch.full((nbytes // 4 + 4,), float("nan"), dtype=torch.float32, device=dev)
        ref_dw = torch.empty_like(dw)
        ref_db = torch.empty_like(db)
        gc.conv_backward_weight(d, xd, gyd, ref_dw, ref_db, ws, nbytes)
        torch.cuda.synchronize()
        assert torch.equal(dw, ref_dw), wl.name
        assert torch.equal(db, ref_db), wl.name


def test_noalloc_rejects_problems_beyond_its_buffer():
    gc.build()
    lib = gc._load()
    limit = gc.conv_backward_weight_noalloc_limit()
    # a wide depthwise layer whose slice partials outgrow the fixed buffer
    C = 1 << 16
    x = gc.geometry((64, C, 64, 64), (64 * 64 * C, 1, 64 * C, C))
    w = gc.geometry((C, 1, 7, 7), (49, 49, 7, 1))
    d = gc.Desc()
    st = (ctypes.c_int32 * 2)(1, 1)
    pd = (ctypes.c_int32 * 2)(3, 3)
    assert lib.conv_bind(ctypes.byref(x), ctypes.byref(w), None, 2, st, pd, pd, None, C,
                         ctypes.byref(d)) == 0
    assert gc.conv_backward_weight_workspace_size(d) > limit
    fake = 1 << 20   # never dereferenced: the size check comes first
    assert lib.conv_backward_weight_noalloc(ctypes.byref(d), fake, fake, fake, None,
                                            None) == 14
    assert "fixed device buffer" in gc.conv_strerror(14)
