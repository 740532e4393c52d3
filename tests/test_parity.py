"""GPU parity: every schedule of the CUDA library against the fp64 oracle.

Each case runs through the C ABI (conv_bind -> out_shape_and_stride ->
conv_dw_forward / conv_grouped_forward) with one schedule forced, and every
output element must satisfy |gpu - ref| <= tol * sum|w*x| + 1e-6 with
tol = 1e-5 (fp32), 2e-3 (fp16), 1.6e-2 (bf16).  Sizes are small enough for
the oracle to finish at once but span several tiles and leave ragged edges.
Schedules that do not apply to a case (the library answers "schedule does
not support this convolution") are skipped for that case; a final test
checks that every schedule ran on some case.
"""

import collections

import numpy as np
import pytest
import torch

import grouped_convolution_gb300 as gc
import oracle
from grouped_convolution_gb300.inputs import ConvWorkload, make_inputs

pytestmark = pytest.mark.gpu

RAN = collections.Counter()

GEOMS = [
    # name, N, Cin_g, Cout_g, G, H, W, KH, KW, stride, pad_before, pad_after
    ("dw3_s1", 2, 1, 1, 48, 13, 11, 3, 3, (1, 1), (1, 1), (1, 1)),
    ("dw3_s2", 2, 1, 1, 32, 17, 19, 3, 3, (2, 2), (1, 1), (1, 1)),
    ("dw7_s1", 1, 1, 1, 40, 15, 18, 7, 7, (1, 1), (3, 3), (3, 3)),
    ("dw5_asym", 1, 1, 1, 24, 20, 23, 5, 5, (2, 1), (2, 0), (1, 3)),
    ("dw9_s1", 1, 1, 1, 16, 12, 13, 9, 9, (1, 1), (4, 4), (4, 4)),
    ("dw1x1", 1, 1, 1, 16, 6, 7, 1, 1, (1, 1), (0, 0), (0, 0)),
    ("dw2x4_s3", 1, 1, 1, 40, 14, 16, 2, 4, (3, 3), (0, 1), (1, 2)),
    ("dw3_c3", 2, 1, 1, 3, 9, 10, 3, 3, (1, 1), (1, 1), (1, 1)),
    ("m4_4x4_same", 2, 1, 4, 8, 15, 14, 4, 4, (1, 1), (1, 1), (2, 2)),
    ("m2_5x3", 1, 1, 2, 12, 11, 17, 5, 3, (1, 2), (2, 1), (2, 1)),
    ("m16_3x3", 1, 1, 16, 4, 9, 9, 3, 3, (1, 1), (1, 1), (1, 1)),
    ("m17_3x3_s2", 1, 1, 17, 3, 8, 8, 3, 3, (2, 2), (1, 1), (1, 1)),
    ("g4x8_9x9_s2", 1, 4, 8, 4, 17, 18, 9, 9, (2, 2), (4, 4), (4, 4)),
    ("g2x3_3x3", 2, 2, 3, 5, 11, 9, 3, 3, (1, 1), (1, 1), (1, 1)),
    ("g8x1_5x5", 1, 8, 1, 2, 10, 10, 5, 5, (1, 1), (2, 2), (2, 2)),
    ("g3x5_4x2", 1, 3, 5, 3, 9, 13, 4, 2, (2, 3), (1, 0), (2, 1)),
    ("g4x8_3x3_many", 1, 4, 8, 16, 20, 20, 3, 3, (1, 1), (1, 1), (1, 1)),
    ("g4x4_7x7", 1, 4, 4, 6, 16, 15, 7, 7, (1, 1), (3, 3), (3, 3)),
    ("g2x2_1x9", 1, 2, 2, 4, 7, 21, 1, 9, (1, 1), (0, 4), (0, 4)),
    ("win_gt_input", 1, 2, 2, 2, 3, 4, 5, 6, (1, 1), (2, 3), (2, 3)),
]

DTYPES = ["f32", "f16", "bf16"]
SCHED = ["dw_flat", "dw_row8", "dw_mult", "grp_plane", "grp_reduce", "grp_tc", "dw_small", "dw_tc",
         "dw_tcl"]


def workload(g, dtype, cl, bias, seed):
    name, N, Cig, Cog, G, H, W, KH, KW, s, pb, pa = g
    return ConvWorkload(name, seed, N=N, C_in=Cig * G, H=H, W=W, C_out=Cog * G, groups=G,
                        KH=KH, KW=KW, stride=s, pad_before=pb, pad_after=pa, dtype=dtype,
                        channels_last=cl, bias=bias)


def run_gpu(wl, x, w, b, schedule, out=None):
    dev = torch.device("cuda")
    xd, wd = x.to(dev), w.to(dev)
    bd = b.to(dev) if b is not None else None
    d = gc.conv_bind(xd, wd, bd, wl.stride, wl.pad_before, wl.pad_after, 1, wl.groups)
    d.schedule = gc.SCHEDULES[schedule]
    y = gc.empty_output(d, xd) if out is None else out
    try:
        name = gc.conv_select_schedule(d, xd, wd, bd, y)
    except gc.GconvError as e:
        if e.status in (7, 11):
            return None
        raise
    assert name == schedule
    fwd = gc.conv_dw_forward if d.Cin_g == 1 else gc.conv_grouped_forward
    fwd(d, xd, wd, bd, y)
    torch.cuda.synchronize()
    return y


def check(wl, x, w, b, y):
    ref, bound = oracle.conv2d(x, w, b, wl.stride, wl.pad_before, wl.pad_after, wl.groups)
    assert tuple(y.shape) == ref.shape
    bad = oracle.violations(y.cpu(), ref, bound, wl.dtype)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        got = y.cpu().double().numpy()
        detail = [(tuple(i), got[tuple(i)], ref[tuple(i)], bound[tuple(i)]) for i in idx]
        pytest.fail(f"{int(bad.sum())}/{bad.size} outside tolerance, e.g. {detail}")


@pytest.mark.parametrize("schedule", SCHED)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cl", [False, True], ids=["nchw", "cl"])
@pytest.mark.parametrize("g", GEOMS, ids=[g[0] for g in GEOMS])
def test_schedule_matches_oracle(g, cl, dtype, schedule):
    bias = (hash(g[0]) + len(dtype)) % 2 == 0
    wl = workload(g, dtype, cl, bias, seed=7 + GEOMS.index(g))
    x, w, b = make_inputs(wl)
    y = run_gpu(wl, x, w, b, schedule)
    if y is None:
        pytest.skip(f"{schedule} does not take this case")
    RAN[schedule] += 1
    check(wl, x, w, b, y)
    # y must be laid out exactly as out_shape_and_stride says
    want = torch.empty(y.shape, device="meta")
    if cl:
        want = want.contiguous(memory_format=torch.channels_last)
    if not (wl.C_out == 1 or y.shape[-1] * y.shape[-2] == 1):
        assert y.stride() == want.stride()


@pytest.mark.parametrize("schedule", SCHED)
@pytest.mark.parametrize("bias", [False, True])
def test_picker_and_bias_flag(schedule, bias):
    g = ("dw3_s1_b", 2, 1, 1, 64, 14, 14, 3, 3, (1, 1), (1, 1), (1, 1))
    wl = workload(g, "bf16", True, bias, seed=99)
    x, w, b = make_inputs(wl)
    y = run_gpu(wl, x, w, b, schedule)
    if y is None:
        pytest.skip("schedule does not take this case")
    check(wl, x, w, b, y)


# dw_mult band geometry: several row bands, several column chunks, every
# window offset against the 16-byte grid (left padding 0..3), row and column
# stride 2 with the band shrunk to fit, multipliers with and without
# 4-channel blocking, rows with and without 16-byte alignment.
MULT_CASES = [
    # name, N, m, C, H, W, KH, KW, stride, pad_before, pad_after
    ("tall_pb0", 1, 4, 3, 300, 30, 3, 3, (1, 1), (1, 0), (1, 3)),
    ("tall_pb1", 1, 4, 3, 290, 40, 4, 4, (1, 1), (1, 1), (2, 2)),
    ("pb2_m3", 2, 3, 2, 61, 48, 5, 5, (1, 1), (2, 2), (2, 2)),
    ("pb3_m8", 1, 8, 2, 40, 53, 7, 7, (1, 1), (3, 3), (3, 3)),
    ("wide_m2", 1, 2, 2, 9, 2100, 3, 9, (1, 1), (1, 4), (1, 4)),
    ("wide_s2", 1, 4, 2, 33, 1504, 3, 3, (2, 2), (1, 1), (1, 1)),
    ("s2_k9_m16", 1, 16, 1, 45, 80, 9, 9, (2, 2), (4, 4), (4, 4)),
    ("s3_1x1", 1, 5, 2, 20, 41, 1, 1, (3, 1), (0, 0), (0, 0)),
]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("case", MULT_CASES, ids=[c[0] for c in MULT_CASES])
def test_dw_mult_geometry_matches_oracle(case, dtype):
    name, N, m, C, H, W, KH, KW, s, pb, pa = case
    wl = ConvWorkload(name, 31 + MULT_CASES.index(case), N=N, C_in=C, H=H, W=W, C_out=C * m,
                      groups=C, KH=KH, KW=KW, stride=s, pad_before=pb, pad_after=pa,
                      dtype=dtype, channels_last=False, bias=m % 2 == 0)
    x, w, b = make_inputs(wl)
    y = run_gpu(wl, x, w, b, "dw_mult")
    assert y is not None, "dw_mult must take this case"
    RAN["dw_mult"] += 1
    check(wl, x, w, b, y)


# grp_tc (tensor-core schedule) tile geometry: several 128-pixel column
# tiles and a ragged last tile, row blocks shorter than a unit, 4 and 8
# input channels per group, 8 / 16 / 32 output channels per 8-channel
# chunk, strides 1 to 3, kernels from 1x1 to 9x9, asymmetric padding, and
# more staged units than CTAs.
TC_CASES = [
    # name, N, Cin_g, Cout_g, G, H, W, KH, KW, stride, pad_before, pad_after
    ("c5_small", 1, 4, 8, 4, 33, 40, 9, 9, (2, 2), (4, 4), (4, 4)),
    ("wide_s1", 1, 4, 4, 2, 7, 150, 3, 3, (1, 1), (1, 1), (1, 1)),
    ("cin8_k5x4", 2, 8, 8, 2, 12, 70, 5, 4, (1, 2), (2, 1), (2, 2)),
    ("cout16_s3", 1, 4, 16, 2, 10, 66, 3, 5, (3, 1), (0, 2), (1, 2)),
    ("k1", 1, 8, 16, 1, 5, 9, 1, 1, (1, 1), (0, 0), (0, 0)),
    ("k9x7_ragged", 1, 4, 8, 2, 20, 129, 9, 7, (2, 2), (4, 3), (4, 3)),
    # several staged units per CTA (more units than CTAs): accumulator
    # blocks reused, weights restaged when a CTA's units change chunk
    ("many_units", 2, 4, 8, 64, 64, 64, 9, 9, (2, 2), (4, 4), (4, 4)),
    ("many_units_2tiles", 2, 8, 16, 32, 24, 160, 3, 3, (1, 1), (1, 1), (1, 1)),
    # the shift form (stride 2, 8 or 16 outputs per chunk): one group per
    # chunk, two column tiles, an even kernel with asymmetric pads, 1x1,
    # many row bands with an odd column pad
    ("s2_cin8", 1, 8, 8, 3, 19, 37, 5, 5, (2, 2), (2, 2), (2, 2)),
    ("s2_wide_ct", 1, 4, 8, 2, 9, 260, 3, 3, (2, 2), (1, 1), (1, 1)),
    ("s2_k4_asym", 2, 4, 8, 4, 14, 22, 4, 4, (2, 2), (1, 1), (2, 2)),
    ("s2_k1", 1, 8, 8, 2, 7, 9, 1, 1, (2, 2), (0, 0), (0, 0)),
    ("s2_tall", 1, 4, 8, 2, 70, 20, 3, 7, (2, 2), (1, 3), (1, 3)),
]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("case", TC_CASES, ids=[c[0] for c in TC_CASES])
def test_grp_tc_geometry_matches_oracle(case, dtype):
    wl = workload(case, dtype, True, TC_CASES.index(case) % 2 == 0, seed=61 + TC_CASES.index(case))
    x, w, b = make_inputs(wl)
    y = run_gpu(wl, x, w, b, "grp_tc")
    assert y is not None, "grp_tc must take this case"
    RAN["grp_tc"] += 1
    check(wl, x, w, b, y)


# dw_tc (NCHW 16-bit depthwise at stride 1 on the tensor cores) geometry:
# multipliers 1 to 16, kernels 1x1 to 9x9 (one and two K steps), every pad
# offset in a chunk, planes taller than a 128-row tile and wider than a unit's
# 128 columns, ragged last tiles, several channels per CTA.
DWTC_CASES = [
    # name, N, Cin_g, Cout_g, G, H, W, KH, KW, stride, pad_before, pad_after
    # (W a multiple of 8: the input rows are TMA boxes of 16-byte chunks)
    ("c4_small", 2, 1, 4, 6, 40, 40, 4, 4, (1, 1), (1, 1), (2, 2)),
    ("m1_k3", 1, 1, 1, 5, 21, 32, 3, 3, (1, 1), (1, 1), (1, 1)),
    ("m2_k9_tall", 1, 1, 2, 2, 150, 24, 9, 9, (1, 1), (4, 4), (4, 4)),
    ("m1_wide", 1, 1, 1, 2, 12, 296, 3, 5, (1, 1), (0, 2), (1, 3)),
    ("m16_k1", 1, 1, 16, 2, 7, 32, 1, 1, (1, 1), (0, 0), (0, 0)),
    ("m8_k7x2_pad7", 1, 1, 8, 2, 11, 24, 7, 2, (1, 1), (3, 7), (3, 0)),
    ("m4_many", 3, 1, 4, 64, 19, 24, 3, 3, (1, 1), (1, 1), (1, 1)),
]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("case", DWTC_CASES, ids=[c[0] for c in DWTC_CASES])
def test_dw_tc_geometry_matches_oracle(case, dtype):
    wl = workload(case, dtype, False, DWTC_CASES.index(case) % 2 == 0, seed=81 + DWTC_CASES.index(case))
    x, w, b = make_inputs(wl)
    y = run_gpu(wl, x, w, b, "dw_tc")
    assert y is not None, "dw_tc must take this case"
    RAN["dw_tc"] += 1
    check(wl, x, w, b, y)


# dw_tcl (channels-last 16-bit depthwise at stride 1 on the tensor cores)
# geometry: several short images stacked in one 128-row tile (a full stack
# and a partial one), images taller than a tile (row blocks), kernels 1x1 to
# 9x9 and 2x8 with every column-tile width, ragged last column tiles,
# asymmetric padding, one channel group per CTA and (past 152 groups) many.
DWTCL_CASES = [
    # name, N, Cin_g, Cout_g, G, H, W, KH, KW, stride, pad_before, pad_after
    # (channels-last, channels a multiple of 8: the input arrives as TMA boxes
    # of 8 channels)
    ("two_images_per_tile", 4, 1, 1, 16, 56, 56, 7, 7, (1, 1), (3, 3), (3, 3)),
    ("row_blocks", 1, 1, 1, 16, 130, 21, 5, 5, (1, 1), (2, 2), (2, 2)),
    ("partial_stack", 5, 1, 1, 8, 9, 40, 7, 7, (1, 1), (3, 3), (3, 3)),
    ("asym_4x6", 2, 1, 1, 24, 17, 30, 4, 6, (1, 1), (1, 2), (2, 3)),
    ("k9_three_blocks", 1, 1, 1, 8, 300, 9, 9, 9, (1, 1), (4, 4), (4, 4)),
    ("k1", 3, 1, 1, 8, 11, 33, 1, 1, (1, 1), (0, 0), (0, 0)),
    ("k2x8_pad7", 2, 1, 1, 8, 64, 19, 2, 8, (1, 1), (0, 7), (1, 0)),
    ("many_groups", 2, 1, 1, 96, 20, 20, 3, 3, (1, 1), (1, 1), (1, 1)),
    ("c96_56x56", 6, 1, 1, 96, 56, 56, 7, 7, (1, 1), (3, 3), (3, 3)),
    # more channel groups than SMs: one contiguous split of all units
    ("groups_past_sm_count", 1, 1, 1, 1232, 9, 12, 3, 3, (1, 1), (1, 1), (1, 1)),
]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("case", DWTCL_CASES, ids=[c[0] for c in DWTCL_CASES])
def test_dw_tcl_geometry_matches_oracle(case, dtype):
    i = DWTCL_CASES.index(case)
    wl = workload(case, dtype, True, i % 2 == 0, seed=131 + i)
    x, w, b = make_inputs(wl)
    y = run_gpu(wl, x, w, b, "dw_tcl")
    assert y is not None, "dw_tcl must take this case"
    RAN["dw_tcl"] += 1
    check(wl, x, w, b, y)


# ------------------------------------------------------------ bit-exact

@pytest.mark.parametrize("schedule", SCHED)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cl", [False, True], ids=["nchw", "cl"])
def test_delta_kernel_bit_exact(schedule, dtype, cl):
    """A one-hot kernel makes every output a copy of one input (or zero in
    the padding): one exact product and exact zeros, so the result is exact."""
    for g in (("d", 2, 1, 2, 16, 11, 12, 4, 5, (1, 2), (2, 1), (1, 3)),
              ("dg", 1, 4, 8, 4, 13, 13, 9, 9, (2, 2), (4, 4), (4, 4)),
              ("d1", 1, 1, 1, 32, 10, 9, 3, 3, (1, 1), (1, 1), (1, 1))):
        wl = workload(g, dtype, cl, False, seed=3)
        x, w, _ = make_inputs(wl)
        KH, KW, Cig = wl.KH, wl.KW, wl.cin_g
        ci0, kh0, kw0 = Cig - 1, KH // 2, KW - 1
        w = torch.zeros_like(w)
        w[:, ci0, kh0, kw0] = 1
        y = run_gpu(wl, x, w, None, schedule)
        if y is None:
            continue
        RAN[schedule] += 1
        got = y.cpu()
        Cog = wl.C_out // wl.groups
        for co in range(wl.C_out):
            c = (co // Cog) * Cig + ci0
            for oh in range(got.shape[2]):
                ih = oh * wl.stride[0] - wl.pad_before[0] + kh0
                for ow in range(got.shape[3]):
                    iw = ow * wl.stride[1] - wl.pad_before[1] + kw0
                    inside = 0 <= ih < wl.H and 0 <= iw < wl.W
                    want = x[:, c, ih, iw] if inside else torch.zeros(wl.N, dtype=x.dtype)
                    assert torch.equal(got[:, co, oh, ow], want), (co, oh, ow)


@pytest.mark.parametrize("schedule", SCHED)
@pytest.mark.parametrize("dtype", DTYPES)
def test_identity_bit_exact(schedule, dtype):
    g = ("id", 2, 1, 1, 24, 9, 11, 1, 1, (1, 1), (0, 0), (0, 0))
    for cl in (False, True):
        wl = workload(g, dtype, cl, False, seed=5)
        x, w, _ = make_inputs(wl)
        w = torch.ones_like(w)
        y = run_gpu(wl, x, w, None, schedule)
        if y is None:
            continue
        assert torch.equal(y.cpu(), x)


@pytest.mark.parametrize("schedule", SCHED)
def test_constant_input_closed_form(schedule):
    """x == 0.5, bf16-exact weights and bias: interior outputs equal
    b + 0.5 * sum(w) up to fp32 rounding of an exact-ish sum."""
    g = ("c", 1, 1, 1, 16, 12, 12, 3, 3, (1, 1), (1, 1), (1, 1))
    wl = workload(g, "f32", True, True, seed=11)
    x, w, b = make_inputs(wl)
    x = torch.full_like(x, 0.5)
    w = torch.round(w * 8) / 8
    b = torch.round(b * 64) / 64
    y = run_gpu(wl, x, w, b, schedule)
    if y is None:
        pytest.skip("schedule does not take this case")
    want = b + 0.5 * w.sum(dim=(1, 2, 3))
    got = y.cpu()[0, :, 5, 5]
    assert torch.equal(got, want)   # all partial sums are exact in fp32


# ---------------------------------------------------------- edge cases

def test_empty_batch_launches_nothing():
    x = torch.empty(0, 8, 9, 9, device="cuda")
    w = torch.randn(8, 1, 3, 3, device="cuda")
    before = gc.conv_launch_count()
    y = gc.conv2d(x, w, None, 1, 1, 1, 8)
    assert y.shape == (0, 8, 9, 9) and gc.conv_launch_count() == before


def test_unbatched_input():
    wl = workload(("u", 1, 1, 1, 8, 9, 9, 3, 3, (1, 1), (1, 1), (1, 1)), "f32", False, True, 13)
    x, w, b = make_inputs(wl)
    y = gc.conv2d(x[0].cuda(), w.cuda(), b.cuda(), 1, 1, 1, 8)
    assert y.shape == (8, 9, 9)
    check(wl, x, w, b, y[None])


@pytest.mark.parametrize("schedule", SCHED)
def test_non_dense_input_and_strided_weights(schedule):
    """A channel slice of a wider channels-last tensor, weights with permuted
    strides and a strided bias."""
    wl = workload(("nd", 2, 1, 1, 16, 10, 11, 3, 3, (1, 1), (1, 1), (1, 1)), "bf16", True, True, 17)
    x, w, b = make_inputs(wl)
    wide = torch.randn(2, 32, 10, 11).to(torch.bfloat16).contiguous(memory_format=torch.channels_last)
    wide[:, 8:24] = x
    wperm = w.permute(0, 2, 3, 1).contiguous().permute(0, 3, 1, 2)
    bwide = torch.zeros(32, dtype=b.dtype)
    bwide[::2] = b
    dev = torch.device("cuda")
    xd, wd, bd = wide.to(dev)[:, 8:24], wperm.to(dev), bwide.to(dev)[::2]
    d = gc.conv_bind(xd, wd, bd, 1, 1, 1, 1, 16)
    assert d.x_dense == 0 and d.layout == 1
    d.schedule = gc.SCHEDULES[schedule]
    y = gc.empty_output(d, xd)
    try:
        gc.conv_select_schedule(d, xd, wd, bd, y)
    except gc.GconvError:
        pytest.skip("schedule does not take non-dense input")
    gc.conv_dw_forward(d, xd, wd, bd, y)
    torch.cuda.synchronize()
    check(wl, x, w, b, y)


@pytest.mark.parametrize("schedule", SCHED)
def test_misaligned_pointers(schedule):
    """Inputs and outputs that start 2 bytes off a 16-byte boundary: the picker
    must avoid vector schedules; a forced vector schedule must refuse."""
    wl = workload(("mis", 1, 1, 1, 16, 9, 9, 3, 3, (1, 1), (1, 1), (1, 1)), "bf16", True, True, 19)
    x, w, b = make_inputs(wl)
    n = x.numel()
    bufx = torch.empty(n + 8, dtype=x.dtype, device="cuda")
    xd = bufx[1:1 + n].view(x.shape[0], x.shape[2], x.shape[3], x.shape[1]).permute(0, 3, 1, 2)
    xd.copy_(x.cuda())
    wd, bd = w.cuda(), b.cuda()
    d = gc.conv_bind(xd, wd, bd, 1, 1, 1, 1, 16)
    sizes, strides = gc.out_shape_and_stride(d)
    bufy = torch.empty(n + 8, dtype=x.dtype, device="cuda")
    y = torch.as_strided(bufy, sizes, strides, 1)
    d.schedule = gc.SCHEDULES[schedule]
    try:
        gc.conv_select_schedule(d, xd, wd, bd, y)
    except gc.GconvError as e:
        assert e.status in (7, 11)
        return
    gc.conv_dw_forward(d, xd, wd, bd, y)
    torch.cuda.synchronize()
    check(wl, x, w, b, y)


@pytest.mark.parametrize("schedule", SCHED)
def test_output_guard_bands_untouched(schedule):
    """Poison the bytes around y; no schedule may write outside y."""
    wl = workload(("gb", 1, 4, 8, 4, 17, 18, 9, 9, (2, 2), (4, 4), (4, 4)), "bf16", True, True, 23)
    x, w, b = make_inputs(wl)
    dev = torch.device("cuda")
    xd, wd, bd = x.to(dev), w.to(dev), b.to(dev)
    d = gc.conv_bind(xd, wd, bd, wl.stride, wl.pad_before, wl.pad_after, 1, wl.groups)
    d.schedule = gc.SCHEDULES[schedule]
    sizes, strides = gc.out_shape_and_stride(d)
    n = int(np.prod(sizes))
    pad = 4096
    buf = torch.full((n + 2 * pad,), 12345.0, dtype=torch.float32, device=dev).to(torch.bfloat16)
    y = torch.as_strided(buf, sizes, strides, pad)
    try:
        gc.conv_select_schedule(d, xd, wd, bd, y)
    except gc.GconvError:
        pytest.skip("schedule does not take this case")
    gc.conv_grouped_forward(d, xd, wd, bd, y)
    torch.cuda.synchronize()
    poison = torch.tensor(12345.0).to(torch.bfloat16)
    assert bool((buf[:pad] == poison).all()) and bool((buf[pad + n:] == poison).all())
    check(wl, x, w, b, y)


CHAIN = [
    # (name, schedule, layout cl, dtype, Cin_g, Cout_g, G, H, W, K, stride)
    ("row8", "dw_row8", True, "bf16", 1, 1, 64, 30, 30, 3, 1),
    ("mult", "dw_mult", False, "f16", 1, 1, 32, 40, 48, 5, 1),
    ("tc", "grp_tc", True, "bf16", 4, 4, 16, 24, 70, 3, 1),
    ("plane", "grp_plane", True, "f32", 4, 4, 8, 20, 20, 3, 1),
    ("flat", "dw_flat", False, "f32", 1, 1, 16, 12, 12, 3, 1),
]


@pytest.mark.parametrize("case", CHAIN, ids=[c[0] for c in CHAIN])
def test_chained_launches_see_previous_output(case):
    """Kernels start early behind the previous launch (programmatic
    dependent launch) but must read its finished output: y2 = conv(conv(x))
    issued back to back many times on one stream, each y2 checked against
    the oracle applied to the y1 the GPU produced."""
    name, sched, cl, dtype, cig, cog, G, H, W, K, s = case
    C = cig * G
    wl = ConvWorkload(name, 91, N=2, C_in=C, H=H, W=W, C_out=C, groups=G, KH=K, KW=K,
                      stride=(s, s), pad_before=(K // 2, K // 2), pad_after=(K // 2, K // 2),
                      dtype=dtype, channels_last=cl, bias=True)
    if cig * G != cog * G:
        pytest.skip("chain needs C_out == C_in")
    x, w, b = make_inputs(wl)
    dev = torch.device("cuda")
    xd, wd, bd = x.to(dev), w.to(dev), b.to(dev)
    pad = K // 2
    outs = []
    for it in range(12):
        y1 = gc.conv2d(xd, wd, bd, s, pad, pad, G, schedule=sched)
        y2 = gc.conv2d(y1, wd, bd, s, pad, pad, G, schedule=sched)
        outs.append((y1, y2))
        xd = y2.clone() if it % 3 == 2 else xd   # feed results forward sometimes
    torch.cuda.synchronize()
    for y1, y2 in outs[-3:]:
        ref, bound = oracle.conv2d(y1.cpu(), w, b, (s, s), (pad, pad), (pad, pad), G)
        bad = oracle.violations(y2.cpu(), ref, bound, dtype)
        assert not bad.any(), f"{int(bad.sum())} outputs differ from the oracle on the GPU's y1"


def test_stream_argument_is_used():
    wl = workload(("st", 1, 1, 1, 16, 9, 9, 3, 3, (1, 1), (1, 1), (1, 1)), "f32", True, True, 29)
    x, w, b = make_inputs(wl)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = gc.conv2d(x.cuda(), w.cuda(), b.cuda(), 1, 1, 1, 16, stream=s)
    s.synchronize()
    check(wl, x, w, b, y)


def test_output_strides_match_torch_cuda_conv():
    """Our output layout rule (dense in the input's format) against what
    torch's CUDA convolution returns for the same call."""
    for cl in (False, True):
        x = torch.randn(2, 16, 12, 12, device="cuda")
        if cl:
            x = x.contiguous(memory_format=torch.channels_last)
        w = torch.randn(32, 1, 3, 3, device="cuda")
        ref = torch.nn.functional.conv2d(x, w, None, 1, 1, 1, 16)
        d = gc.conv_bind(x, w, None, 1, 1, 1, 1, 16)
        sizes, strides = gc.out_shape_and_stride(d)
        assert sizes == tuple(ref.shape)
        assert strides == tuple(ref.stride())


def test_every_schedule_ran():
    """Collected last in this file: each schedule took at least one case."""
    missing = [s for s in SCHED if RAN[s] == 0]
    assert not missing, f"schedules never exercised: {missing}"
