"""GPU parity for the wider envelope: dilated and 1-D forward convolutions,
transposed convolutions (executorch PR #25091, description, second
paragraph) and the backward (dx, dw, db), against the fp64 oracle.

Every case runs through the C ABI with each schedule that takes it forced in
turn (plus the picker's choice), and every output element must satisfy
|gpu - ref| <= tol * bound + 1e-6 with the oracle's bound (sum of |terms|).
Sizes span several blocks and leave ragged edges; layouts, dtypes, strides,
dilations, asymmetric paddings and crops, output_padding and multipliers
vary across the cases.
"""

import collections

import numpy as np
import pytest
import torch

import grouped_convolution_gb300 as gc
import oracle
from grouped_convolution_gb300.inputs import ConvWorkload, make_grad, make_inputs

pytestmark = pytest.mark.gpu

RAN = collections.Counter()
DTYPES = ["f32", "f16", "bf16"]
SCHED = ["auto", "dw_flat", "grp_reduce", "dw_line", "dw_row8", "dw_mult", "grp_plane"]


def wl_of(case, dtype, cl, bias, seed, **kw):
    name, N, Cig, Cog, G, H, W, KH, KW, s, pb, pa = case[:12]
    return ConvWorkload(name, seed, N=N, C_in=Cig * G, H=H, W=W, C_out=Cog * G, groups=G,
                        KH=KH, KW=KW, stride=s, pad_before=pb, pad_after=pa, dtype=dtype,
                        channels_last=cl, bias=bias, **kw)


def gpu_run(wl, x, w, b, schedule):
    dev = torch.device("cuda")
    xd, wd = x.to(dev), w.to(dev)
    bd = b.to(dev) if b is not None else None
    d = gc.bind(xd, wd, bd, wl.stride, wl.pad_before, wl.pad_after, wl.dilation, wl.groups,
                wl.transposed, wl.output_padding)
    d.schedule = gc.SCHEDULES[schedule]
    y = gc.empty_output(d, xd)
    try:
        name = gc.conv_select_schedule(d, xd, wd, bd, y)
    except gc.GconvError as e:
        if e.status in (7, 11):
            return None, None
        raise
    if schedule != "auto":
        assert name == schedule
    gc.run(d, xd, wd, bd, y)
    torch.cuda.synchronize()
    return y, name


def check(y, ref, bound, dtype):
    assert tuple(y.shape) == ref.shape
    bad = oracle.violations(y.cpu(), ref, bound, dtype)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        got = y.cpu().double().numpy()
        detail = [(tuple(i), got[tuple(i)], ref[tuple(i)], bound[tuple(i)]) for i in idx]
        pytest.fail(f"{int(bad.sum())}/{bad.size} outside tolerance, e.g. {detail}")


# ---------------------------------------------------------- dilated forward

DIL = [
    # name, N, Cig, Cog, G, H, W, KH, KW, stride, pb, pa, dilation
    ("dw3_d2", 2, 1, 1, 48, 15, 13, 3, 3, (1, 1), (2, 2), (2, 2), (2, 2)),
    ("dw3_d3_s2", 1, 1, 1, 40, 21, 19, 3, 3, (2, 2), (3, 1), (3, 4), (3, 3)),
    ("dw5x3_d21", 1, 1, 1, 32, 17, 23, 5, 3, (1, 2), (4, 2), (4, 0), (2, 1)),
    ("m2_3x3_d2", 1, 1, 2, 16, 12, 12, 3, 3, (1, 1), (2, 2), (2, 2), (2, 2)),
    ("g4x8_3x3_d2", 1, 4, 8, 4, 14, 15, 3, 3, (1, 1), (2, 2), (2, 2), (2, 2)),
    ("dw9_d2", 1, 1, 1, 16, 20, 20, 9, 9, (1, 1), (8, 8), (8, 8), (2, 2)),
    # dw_row8's dilated ring (3x3, dilation 2, stride 1): long runs with
    # asymmetric pads, two channel chunks
    ("dw3_d2_tall", 4, 1, 1, 16, 60, 21, 3, 3, (1, 1), (2, 1), (1, 2), (2, 2)),
    ("dw3_d2_c264", 1, 1, 1, 264, 9, 10, 3, 3, (1, 1), (2, 2), (2, 2), (2, 2)),
]


@pytest.mark.parametrize("schedule", SCHED)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cl", [False, True], ids=["nchw", "cl"])
@pytest.mark.parametrize("case", DIL, ids=[c[0] for c in DIL])
def test_dilated_forward(case, cl, dtype, schedule):
    wl = wl_of(case, dtype, cl, DIL.index(case) % 2 == 0, 300 + DIL.index(case),
               dilation=case[12])
    x, w, b = make_inputs(wl)
    y, name = gpu_run(wl, x, w, b, schedule)
    if y is None:
        pytest.skip(f"{schedule} does not take this case")
    RAN[("dil", name)] += 1
    ref, bound = oracle.reference(wl, x, w, b)
    check(y, ref, bound, dtype)


# ---------------------------------------------------------------------- 1-D

ONED = [
    # name, N, Cig, Cog, G, 1, L, 1, K, (1, s), (0, pb), (0, pa), dilation
    ("causal_k4", 2, 1, 1, 64, 1, 100, 1, 4, (1, 1), (0, 3), (0, 0), (1, 1)),
    ("k7_s2", 3, 1, 1, 40, 1, 77, 1, 7, (1, 2), (0, 3), (0, 3), (1, 1)),
    ("k3_d4", 1, 1, 1, 24, 1, 65, 1, 3, (1, 1), (0, 4), (0, 4), (1, 4)),
    ("k9_m3", 1, 1, 3, 8, 1, 50, 1, 9, (1, 1), (0, 8), (0, 0), (1, 1)),
    ("g4x4_k5", 1, 4, 4, 6, 1, 45, 1, 5, (1, 3), (0, 2), (0, 2), (1, 1)),
]


@pytest.mark.parametrize("schedule", SCHED)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cl", [False, True], ids=["ncl", "nlc"])
@pytest.mark.parametrize("case", ONED, ids=[c[0] for c in ONED])
def test_conv1d(case, cl, dtype, schedule):
    wl = wl_of(case, dtype, cl, True, 400 + ONED.index(case), dilation=case[12],
               spatial_dims=1)
    x, w, b = make_inputs(wl)
    y, name = gpu_run(wl, x, w, b, schedule)
    if y is None:
        pytest.skip(f"{schedule} does not take this case")
    RAN[("1d", name)] += 1
    assert y.dim() == 3
    ref, bound = oracle.reference(wl, x, w, b)
    check(y, ref, bound, dtype)


def test_conv1d_unbatched_and_strides():
    wl = wl_of(ONED[0], "bf16", True, True, 450, spatial_dims=1)
    x, w, b = make_inputs(wl.replace(N=1))
    xd = x[0].cuda()                     # [C, L], channels-last order (C stride 1)
    y = gc.conv1d(xd, w.cuda(), b.cuda(), 1, 3, 0, wl.groups)
    torch.cuda.synchronize()
    assert y.dim() == 2 and y.stride() == (1, wl.C_out)
    ref, bound = oracle.conv1d(x[0], w, b, 1, 3, 0, wl.groups)
    check(y, ref[0], bound[0], "bf16")


# --------------------------------------------------------------- transposed

TR = [
    # name, N, Cig, Cog, G, H, W, KH, KW, stride, crop_before, crop_after, out_pad, dil
    ("dw4_s2_up", 2, 1, 1, 48, 9, 11, 4, 4, (2, 2), (1, 1), (1, 1), (0, 0), (1, 1)),
    ("dw3_s2_op1", 1, 1, 1, 40, 8, 7, 3, 3, (2, 2), (1, 1), (1, 1), (1, 1), (1, 1)),
    ("dw3_s1", 2, 1, 1, 32, 10, 12, 3, 3, (1, 1), (1, 1), (1, 1), (0, 0), (1, 1)),
    ("dw5_s1_asym", 1, 1, 1, 24, 9, 13, 5, 5, (1, 1), (3, 1), (0, 4), (0, 0), (1, 1)),
    ("dw3_s1_bigcrop", 1, 1, 1, 16, 12, 12, 3, 3, (1, 1), (3, 0), (0, 3), (0, 0), (1, 1)),
    ("dw3_s3_d2", 1, 1, 1, 16, 7, 6, 3, 3, (3, 3), (2, 0), (0, 2), (2, 1), (2, 2)),
    ("m2_4x4_s2", 1, 1, 2, 8, 6, 7, 4, 4, (2, 2), (1, 1), (1, 1), (0, 0), (1, 1)),
    ("m3_3x3_s1", 1, 1, 3, 8, 7, 9, 3, 3, (1, 1), (1, 1), (1, 1), (0, 0), (1, 1)),
    ("g4x2_3x3_s2", 1, 4, 2, 4, 8, 8, 3, 3, (2, 2), (1, 1), (1, 1), (1, 1), (1, 1)),
    ("g8x8_5x5_s1", 1, 8, 8, 2, 9, 10, 5, 5, (1, 1), (2, 2), (2, 2), (0, 0), (1, 1)),
    ("g4x1_3x3_s1", 2, 4, 1, 6, 9, 10, 3, 3, (1, 1), (1, 0), (1, 2), (0, 1), (1, 1)),
    ("g8x1_4x2_s1_d2", 1, 8, 1, 3, 8, 7, 4, 2, (1, 1), (3, 1), (2, 0), (0, 0), (2, 1)),
    # stride-2 depthwise square kernels: long runs, odd and even crops, two
    # channel chunks, with and without bias
    ("dw3_s2_tall", 4, 1, 1, 16, 40, 21, 3, 3, (2, 2), (0, 0), (0, 0), (0, 0), (1, 1)),
    ("dw5_s2_odd", 2, 1, 1, 24, 17, 30, 5, 5, (2, 2), (1, 1), (2, 1), (1, 0), (1, 1)),
    ("dw7_s2_c264", 1, 1, 1, 264, 6, 9, 7, 7, (2, 2), (3, 2), (2, 3), (1, 1), (1, 1)),
    ("dw3_s2_c264", 2, 1, 1, 264, 9, 8, 3, 3, (2, 2), (1, 1), (1, 1), (1, 1), (1, 1)),
]


@pytest.mark.parametrize("schedule", SCHED)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cl", [False, True], ids=["nchw", "cl"])
@pytest.mark.parametrize("case", TR, ids=[c[0] for c in TR])
def test_transposed(case, cl, dtype, schedule):
    wl = wl_of(case, dtype, cl, TR.index(case) % 2 == 1, 500 + TR.index(case),
               transposed=True, output_padding=case[12], dilation=case[13])
    x, w, b = make_inputs(wl)
    y, name = gpu_run(wl, x, w, b, schedule)
    if y is None:
        pytest.skip(f"{schedule} does not take this case")
    RAN[("tr", name)] += 1
    ref, bound = oracle.reference(wl, x, w, b)
    check(y, ref, bound, dtype)


@pytest.mark.parametrize("cl", [False, True], ids=["ncl", "nlc"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_transposed_1d_upsampling(cl, dtype):
    case = ("up_k4_s2", 2, 1, 1, 64, 1, 70, 1, 4, (1, 2), (0, 1), (0, 1))
    wl = wl_of(case, dtype, cl, True, 560, transposed=True, spatial_dims=1)
    x, w, b = make_inputs(wl)
    for schedule in ("auto", "dw_line", "dw_flat", "grp_reduce"):
        y, name = gpu_run(wl, x, w, b, schedule)
        if y is None:
            continue
        RAN[("tr1d", name)] += 1
        assert y.dim() == 3 and y.shape[-1] == 140
        ref, bound = oracle.reference(wl, x, w, b)
        check(y, ref, bound, dtype)


# ----------------------------------------------------------------- backward

BWD = [
    # name, N, Cig, Cog, G, H, W, KH, KW, stride, pb, pa, dilation
    ("dw3_s1", 2, 1, 1, 48, 13, 11, 3, 3, (1, 1), (1, 1), (1, 1), (1, 1)),
    ("dw3_s2", 2, 1, 1, 32, 15, 16, 3, 3, (2, 2), (1, 1), (1, 1), (1, 1)),
    ("dw7_s1", 1, 1, 1, 24, 14, 15, 7, 7, (1, 1), (3, 3), (3, 3), (1, 1)),
    ("dw5_s2_rem", 1, 1, 1, 16, 12, 13, 5, 5, (2, 2), (2, 1), (0, 2), (1, 1)),
    ("dw3_d2", 1, 1, 1, 40, 12, 12, 3, 3, (1, 1), (2, 2), (2, 2), (2, 2)),
    ("m4_4x4", 2, 1, 4, 8, 11, 10, 4, 4, (1, 1), (1, 1), (2, 2), (1, 1)),
    ("g4x8_9x9_s2", 1, 4, 8, 4, 17, 18, 9, 9, (2, 2), (4, 4), (4, 4), (1, 1)),
    ("g2x3_3x3", 2, 2, 3, 5, 9, 9, 3, 3, (1, 1), (1, 1), (1, 1), (1, 1)),
    ("dw1x7_s1", 2, 1, 1, 40, 5, 30, 1, 7, (1, 1), (0, 3), (0, 3), (1, 1)),
    ("dw2x2_s1_ragged", 3, 1, 1, 24, 7, 13, 2, 2, (2, 1), (0, 1), (1, 0), (1, 1)),
    ("dw1x3_d3", 1, 1, 1, 32, 4, 29, 1, 3, (1, 1), (0, 3), (0, 3), (1, 3)),
    ("dw2x3_sw2_ragged", 2, 1, 1, 144, 6, 23, 2, 3, (1, 2), (1, 0), (0, 2), (1, 1)),
    ("dw1x5_sw2", 2, 1, 1, 40, 3, 37, 1, 5, (1, 2), (0, 2), (0, 1), (1, 1)),
    ("dw3_s2_d2", 1, 1, 1, 24, 11, 17, 3, 3, (2, 2), (2, 2), (2, 2), (2, 2)),
    # long runs of output rows per CTA, both strides; two channel chunks
    ("dw3_s1_tall", 8, 1, 1, 16, 160, 20, 3, 3, (1, 1), (1, 1), (1, 1), (1, 1)),
    ("dw3_s2_tall", 8, 1, 1, 16, 161, 21, 3, 3, (2, 2), (1, 0), (0, 1), (1, 1)),
    ("dw3_s1_c264", 1, 1, 1, 264, 6, 7, 3, 3, (1, 1), (1, 1), (1, 1), (1, 1)),
    ("dw7_s1_tall", 4, 1, 1, 16, 70, 20, 7, 7, (1, 1), (3, 3), (3, 3), (1, 1)),
    ("dw5_s2_tall", 4, 1, 1, 16, 81, 30, 5, 5, (2, 2), (2, 2), (2, 2), (1, 1)),
    ("dw7_s2_ragged", 2, 1, 1, 24, 23, 19, 7, 7, (2, 2), (3, 2), (2, 3), (1, 1)),
]


def bwd_inputs(case, dtype, cl, seed):
    wl = wl_of(case, dtype, cl, False, seed, dilation=case[12])
    x, w, _ = make_inputs(wl)
    ref, _ = oracle.reference(wl, x, w, None)
    gy = make_grad(wl, ref.shape)
    return wl, x, w, gy


@pytest.mark.parametrize("schedule", SCHED)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cl", [False, True], ids=["nchw", "cl"])
@pytest.mark.parametrize("case", BWD, ids=[c[0] for c in BWD])
def test_backward_input(case, cl, dtype, schedule):
    wl, x, w, gy = bwd_inputs(case, dtype, cl, 600 + BWD.index(case))
    dev = torch.device("cuda")
    xd, wd, gyd = x.to(dev), w.to(dev), gy.to(dev)
    d = gc.conv_bind(xd, wd, None, wl.stride, wl.pad_before, wl.pad_after, wl.dilation,
                     wl.groups)
    d.schedule = gc.SCHEDULES[schedule]
    sizes, strides = gc.grad_input_shape_and_stride(d)
    assert tuple(sizes) == tuple(x.shape)
    dx = torch.empty_strided(sizes, strides, dtype=x.dtype, device=dev)
    try:
        gc.conv_backward_input(d, gyd, wd, dx)
    except gc.GconvError as e:
        if e.status in (7, 11):
            pytest.skip(f"{schedule} does not take this case")
        raise
    torch.cuda.synchronize()
    RAN[("dx", schedule)] += 1
    g = oracle.conv2d_backward(x, w, gy, wl.stride, wl.pad_before, wl.pad_after, wl.groups,
                               wl.dilation, need=("dx",))
    check(dx, g["dx"][0], g["dx"][1], dtype)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cl", [False, True], ids=["nchw", "cl"])
@pytest.mark.parametrize("case", BWD, ids=[c[0] for c in BWD])
def test_backward_weight_and_bias(case, cl, dtype):
    wl, x, w, gy = bwd_inputs(case, dtype, cl, 700 + BWD.index(case))
    dev = torch.device("cuda")
    xd, wd, gyd = x.to(dev), w.to(dev), gy.to(dev)
    out = gc.conv2d_backward(xd, wd, gyd, wl.stride, wl.pad_before, wl.pad_after, wl.groups,
                             wl.dilation, need=("dw", "db"))
    torch.cuda.synchronize()
    g = oracle.conv2d_backward(x, w, gy, wl.stride, wl.pad_before, wl.pad_after, wl.groups,
                               wl.dilation, need=("dw", "db"))
    check(out["dw"], g["dw"][0], g["dw"][1], dtype)
    check(out["db"], g["db"][0], g["db"][1], dtype)
    # deterministic: a second run gives the same bits
    again = gc.conv2d_backward(xd, wd, gyd, wl.stride, wl.pad_before, wl.pad_after, wl.groups,
                               wl.dilation, need=("dw", "db"))
    torch.cuda.synchronize()
    assert torch.equal(again["dw"], out["dw"]) and torch.equal(again["db"], out["db"])


def test_backward_weight_workspace_contract():
    case = BWD[0]
    wl, x, w, gy = bwd_inputs(case, "bf16", True, 790)
    dev = torch.device("cuda")
    xd, wd, gyd = x.to(dev), w.to(dev), gy.to(dev)
    d = gc.conv_bind(xd, wd, None, wl.stride, wl.pad_before, wl.pad_after, 1, wl.groups)
    need = gc.conv_backward_weight_workspace_size(d)
    dw = torch.empty(tuple(w.shape), dtype=w.dtype, device=dev)
    ws = torch.empty(need // 4 + 4, dtype=torch.float32, device=dev)
    with pytest.raises(gc.GconvError) as e:
        gc.conv_backward_weight(d, xd, gyd, dw, None, ws, need - 4)
    assert e.value.status == 13
    # stale workspace contents do not matter: fill with NaN, result stays exact
    ws.fill_(float("nan"))
    gc.conv_backward_weight(d, xd, gyd, dw, None, ws, need)
    torch.cuda.synchronize()
    g = oracle.conv2d_backward(x, w, gy, wl.stride, wl.pad_before, wl.pad_after, wl.groups,
                               need=("dw",))
    check(dw, g["dw"][0], g["dw"][1], "bf16")


def test_backward_empty_batch_gives_zero_weight_grad():
    case = BWD[0]
    wl, x, w, gy = bwd_inputs(case, "f32", True, 791)
    dev = torch.device("cuda")
    x0 = x[:0].to(dev)
    gy0 = gy[:0].to(dev)
    out = gc.conv2d_backward(x0, w.to(dev), gy0, wl.stride, wl.pad_before, wl.pad_after,
                             wl.groups, need=("dx", "dw", "db"))
    torch.cuda.synchronize()
    assert out["dx"].shape[0] == 0
    assert torch.count_nonzero(out["dw"]) == 0 and torch.count_nonzero(out["db"]) == 0


def test_every_new_path_ran():
    # the transposed stride-1 one-channel-per-group cases must have run as a
    # flipped forward on a forward schedule, the others on dw_line / dw_flat /
    # grp_reduce
    names = {k[1] for k in RAN}
    for want in ("dw_flat", "grp_reduce", "dw_line", "dw_row8"):
        assert want in names, (want, dict(RAN))


# ------------------------------------------------- alignment and guard bands

def _offset_copy(t, elems=1, pad=8):
    """t copied into a buffer at an element offset (breaks 16-byte
    alignment), keeping t's strides."""
    n = t.untyped_storage().nbytes() // t.element_size()
    buf = torch.empty(n + pad, dtype=t.dtype, device="cuda")
    out = torch.as_strided(buf, t.shape, t.stride(), elems)
    out.copy_(t.cuda())
    return out


@pytest.mark.parametrize("schedule", ["auto", "dw_line", "dw_flat", "grp_reduce"])
def test_transposed_misaligned_input(schedule):
    case = ("mis_up", 2, 1, 1, 32, 9, 11, 4, 4, (2, 2), (1, 1), (1, 1))
    wl = wl_of(case, "bf16", True, True, 810, transposed=True)
    x, w, b = make_inputs(wl)
    xd = _offset_copy(x)
    wd, bd = w.cuda(), b.cuda()
    d = gc.bind(xd, wd, bd, wl.stride, wl.pad_before, wl.pad_after, 1, wl.groups, True, 0)
    d.schedule = gc.SCHEDULES[schedule]
    y = gc.empty_output(d, xd)
    try:
        name = gc.conv_select_schedule(d, xd, wd, bd, y)
    except gc.GconvError as e:
        assert schedule == "dw_line" and e.status == 7   # needs 16-byte alignment
        return
    assert name != "dw_line"
    gc.run(d, xd, wd, bd, y)
    torch.cuda.synchronize()
    ref, bound = oracle.reference(wl, x, w, b)
    check(y, ref, bound, "bf16")


def test_backward_misaligned_and_guard_bands():
    case = BWD[0]
    wl, x, w, gy = bwd_inputs(case, "bf16", True, 820)
    dev = torch.device("cuda")
    xd, gyd, wd = _offset_copy(x), _offset_copy(gy), w.to(dev)
    d = gc.conv_bind(xd, wd, None, wl.stride, wl.pad_before, wl.pad_after, 1, wl.groups)
    g = oracle.conv2d_backward(x, w, gy, wl.stride, wl.pad_before, wl.pad_after, wl.groups)
    pad = 2048
    poison = torch.tensor(777.0).to(torch.bfloat16)
    # dx into a guarded buffer
    sizes, strides = gc.grad_input_shape_and_stride(d)
    n = int(np.prod(sizes))
    bufx = torch.full((n + 2 * pad,), 777.0, device=dev).to(torch.bfloat16)
    dx = torch.as_strided(bufx, sizes, strides, pad)
    gc.conv_backward_input(d, gyd, wd, dx)
    # dw / db into guarded buffers; the misaligned x and gy take the generic form
    nw = w.numel()
    bufw = torch.full((nw + 2 * pad,), 777.0, device=dev).to(torch.bfloat16)
    dw = torch.as_strided(bufw, tuple(w.shape), w.stride(), pad)
    bufb = torch.full((d.C_out + 2 * pad,), 777.0, device=dev).to(torch.bfloat16)
    db = torch.as_strided(bufb, (d.C_out,), (1,), pad)
    nbytes = gc.conv_backward_weight_workspace_size(d)
    ws = torch.empty(nbytes // 4 + 4, dtype=torch.float32, device=dev)
    gc.conv_backward_weight(d, xd, gyd, dw, db, ws, nbytes)
    torch.cuda.synchronize()
    for buf, m in ((bufx, n), (bufw, nw), (bufb, d.C_out)):
        assert bool((buf[:pad] == poison).all()) and bool((buf[pad + m:] == poison).all())
    check(dx, g["dx"][0], g["dx"][1], "bf16")
    check(dw, g["dw"][0], g["dw"][1], "bf16")
    check(db, g["db"][0], g["db"][1], "bf16")


@pytest.mark.parametrize("kind", ["dilated", "causal_1d", "transposed"])
def test_dw_line_output_guard_bands(kind):
    if kind == "dilated":
        wl = wl_of(DIL[0], "bf16", True, True, 830, dilation=DIL[0][12])
    elif kind == "causal_1d":
        wl = wl_of(ONED[0], "bf16", True, True, 831, spatial_dims=1)
    else:
        wl = wl_of(TR[0], "bf16", True, True, 832, transposed=True)
    x, w, b = make_inputs(wl)
    dev = torch.device("cuda")
    xd, wd, bd = x.to(dev), w.to(dev), b.to(dev)
    d = gc.bind(xd, wd, bd, wl.stride, wl.pad_before, wl.pad_after, wl.dilation, wl.groups,
                wl.transposed, wl.output_padding)
    d.schedule = gc.SCHEDULES["dw_line"]
    sizes, strides = gc.out_shape_and_stride(d)
    n = int(np.prod(sizes))
    pad = 4096
    buf = torch.full((n + 2 * pad,), 777.0, device=dev).to(torch.bfloat16)
    y = torch.as_strided(buf, sizes, strides, pad)
    gc.run(d, xd, wd, bd, y)
    torch.cuda.synchronize()
    poison = torch.tensor(777.0).to(torch.bfloat16)
    assert bool((buf[:pad] == poison).all()) and bool((buf[pad + n:] == poison).all())
    ref, bound = oracle.reference(wl, x, w, b)
    check(y, ref, bound, "bf16")
