"""Host logic of the C ABI, on the CPU: binding and validation, layout
detection, the output shape/stride rule, schedule selection and the failure
contract.  Nothing here launches a kernel (fake, aligned device addresses are
only inspected), so no GPU is needed."""

import itertools

import pytest
import torch

import grouped_convolution_gb300 as gc
import oracle
from grouped_convolution_gb300.inputs import WORKLOADS

ERR = {"NULL": 1, "RANK": 2, "DTYPE": 3, "SHAPE": 4, "UNSUPPORTED": 5, "PADDING": 6,
       "ALIGN": 7, "CUDA": 8, "INTERNAL": 9, "LAYOUT": 10, "SCHEDULE": 11, "KIND": 12,
       "WORKSPACE": 13}

FAKE = 1 << 20   # a 1 MiB-aligned fake device address; never dereferenced


@pytest.fixture(scope="module", autouse=True)
def lib():
    gc.build()
    yield
    gc.conv_force_schedule("auto")


def geo(shape, strides=None):
    if strides is None:   # dense, row-major
        strides, acc = [], 1
        for n in reversed(shape):
            strides.insert(0, acc)
            acc *= max(n, 1)
    return (tuple(shape), tuple(strides))


def cl_strides(N, C, H, W):
    return (H * W * C, 1, W * C, C)


def bind(x=((1, 4, 8, 8), None), w=((4, 1, 3, 3), None), b=None, stride=1, pb=1, pa=None,
         dil=1, groups=4, dtype="float32"):
    xg = geo(*x) if x is not None else None
    wg = geo(*w) if w is not None else None
    bg = geo(*b) if b is not None else None
    return gc.conv_bind(xg, wg, bg, stride, pb, pa, dil, groups, dtype=dtype)


def status_of(fn):
    try:
        fn()
    except gc.GconvError as e:
        return e.status
    return 0


# ---------------------------------------------------------------- validation

def test_valid_depthwise_desc():
    d = bind(b=((4,), None))
    assert (d.N, d.C_in, d.H, d.W, d.C_out, d.groups, d.Cin_g, d.Cout_g) == (1, 4, 8, 8, 4, 4, 1, 1)
    assert (d.KH, d.KW, d.OH, d.OW) == (3, 3, 8, 8)
    assert d.has_bias == 1 and d.layout == 0 and d.unbatched == 0 and d.schedule == -1
    assert list(d.pad_before) == [1, 1] and list(d.pad_after) == [1, 1]
    assert d.x_dense == 1


@pytest.mark.parametrize("kw,err", [
    (dict(groups=3), "SHAPE"),                               # C_in % groups
    (dict(w=((4, 2, 3, 3), None), groups=4), "SHAPE"),      # Cin_g * groups != C_in
    (dict(w=((6, 1, 3, 3), None), groups=4), "SHAPE"),      # C_out % groups
    (dict(b=((5,), None)), "SHAPE"),                         # bias size
    (dict(stride=0), "SHAPE"),
    (dict(groups=0), "SHAPE"),
    (dict(dil=0), "UNSUPPORTED"),
    (dict(dil=4, pb=0, pa=0), "PADDING"),                    # dilated span 9 > 8
    (dict(w=((4, 1, 10, 3), None)), "UNSUPPORTED"),          # KH > 9
    (dict(w=((4, 1, 3, 10), None)), "UNSUPPORTED"),          # KW > 9
    (dict(x=((1, 9, 8, 8), None), w=((9, 9, 3, 3), None), groups=1), "UNSUPPORTED"),  # Cin_g 9
    (dict(pb=-1), "PADDING"),
    (dict(pb=0, pa=0, w=((4, 1, 9, 3), None)), "PADDING"),   # window taller than input
    (dict(x=((4, 8, 8), None), w=((4, 1, 3), None)), "RANK"),
    (dict(x=((1, 1, 4, 8, 8), None)), "RANK"),
    (dict(b=((1, 4), None)), "RANK"),
    (dict(x=((1, 4, 8, 8), (256, 1, 8, 32))), "LAYOUT"),     # (N, C, W, H) order
    (dict(x=((1, 4, 8, 8), (256, 64, 8, 2))), "LAYOUT"),     # W stride 2, no stride-1 dim
    (dict(x=((1, 4, 8, 8), (256, 32, 8, 1))), "LAYOUT"),     # overlapping C / H
])
def test_rejections(kw, err):
    assert status_of(lambda: bind(**kw)) == ERR[err]


def test_bad_dtype_and_nulls():
    lib = gc._load()
    d = gc.Desc()
    x = gc.geometry((1, 4, 8, 8), (256, 64, 8, 1))
    w = gc.geometry((4, 1, 3, 3), (9, 9, 3, 1))
    import ctypes
    assert lib.conv_bind(ctypes.byref(x), ctypes.byref(w), None, 7, None, None, None, None, 4,
                         ctypes.byref(d)) == ERR["DTYPE"]
    assert lib.conv_bind(None, ctypes.byref(w), None, 0, None, None, None, None, 4,
                         ctypes.byref(d)) == ERR["NULL"]
    assert lib.conv_bind(ctypes.byref(x), ctypes.byref(w), None, 0, None, None, None, None, 4,
                         None) == ERR["NULL"]
    # NULL scalars take the canonical defaults: stride 1, padding 0, dilation 1.
    assert lib.conv_bind(ctypes.byref(x), ctypes.byref(w), None, 0, None, None, None, None, 4,
                         ctypes.byref(d)) == 0
    assert (d.OH, d.OW, list(d.stride), list(d.pad_before), list(d.pad_after)) == (
        6, 6, [1, 1], [0, 0], [0, 0])


def test_unbatched_input():
    d = bind(x=((4, 8, 8), None))
    assert d.unbatched == 1 and d.N == 1
    sizes, strides = gc.out_shape_and_stride(d)
    assert sizes == (4, 8, 8) and strides == (64, 8, 1)


def test_uninitialised_desc_is_rejected():
    d = gc.Desc()
    assert status_of(lambda: gc.out_shape_and_stride(d)) == ERR["INTERNAL"]
    assert status_of(lambda: gc.conv_dw_forward(d, FAKE, FAKE, None, FAKE, 0)) == ERR["INTERNAL"]


# ------------------------------------------------------------------- layout

def test_layout_detection():
    N, C, H, W = 2, 6, 5, 7
    d = bind(x=((N, C, H, W), cl_strides(N, C, H, W)), w=((C, 1, 3, 3), None), groups=C)
    assert d.layout == 1 and d.x_dense == 1
    d = bind(x=((N, C, H, W), None), w=((C, 1, 3, 3), None), groups=C)
    assert d.layout == 0 and d.x_dense == 1
    # C == 1: both orders fit; NCHW is taken.
    d = bind(x=((N, 1, H, W), (H * W, H * W, W, 1)), w=((3, 1, 3, 3), None), groups=1)
    assert d.layout == 0
    # Ordered but not dense (a channel slice of a channels-last tensor).
    big = cl_strides(N, 2 * C, H, W)
    d = bind(x=((N, C, H, W), big), w=((C, 1, 3, 3), None), groups=C)
    assert d.layout == 1 and d.x_dense == 0


def test_weight_and_bias_strides_are_free():
    w = torch.empty(8, 3, 3, 4).permute(0, 3, 1, 2)   # [8, 4, 3, 3] with odd strides
    d = bind(x=((1, 8, 9, 9), None), w=(tuple(w.shape), tuple(w.stride())), groups=2,
             b=((8,), (3,)))
    assert tuple(d.w_strides) == tuple(w.stride()) and d.b_stride == 3


# --------------------------------------------------------- output shape rule

@pytest.mark.parametrize("H,K,s,pb,pa", list(itertools.product(
    [1, 3, 8, 56, 57], [1, 2, 3, 4, 7, 9], [1, 2, 3], [0, 1, 4], [0, 2, 3])))
def test_out_shape_matches_oracle(H, K, s, pb, pa):
    want = oracle.out_size(H, K, s, pb, pa)
    call = lambda: bind(x=((1, 2, H, H + 1), None), w=((2, 1, K, K), None), groups=2,
                        stride=s, pb=pb, pa=pa)
    if want < 0:
        assert status_of(call) == ERR["PADDING"]
        return
    d = call()
    sizes, strides = gc.out_shape_and_stride(d)
    assert sizes == (1, 2, want, oracle.out_size(H + 1, K, s, pb, pa))


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workload_output_geometry(name):
    wl = WORKLOADS[name]
    x = torch.empty(wl.N, wl.C_in, wl.H, wl.W, device="meta")
    if wl.channels_last:
        x = x.contiguous(memory_format=torch.channels_last)
    d = gc.conv_bind((tuple(x.shape), tuple(x.stride())),
                     ((wl.C_out, wl.cin_g, wl.KH, wl.KW), (wl.cin_g * wl.KH * wl.KW, wl.KH * wl.KW, wl.KW, 1)),
                     ((wl.C_out,), (1,)) if wl.bias else None, wl.stride, wl.pad_before,
                     wl.pad_after, 1, wl.groups, dtype=str(wl.torch_dtype))
    sizes, strides = gc.out_shape_and_stride(d)
    OH = oracle.out_size(wl.H, wl.KH, wl.stride[0], wl.pad_before[0], wl.pad_after[0])
    OW = oracle.out_size(wl.W, wl.KW, wl.stride[1], wl.pad_before[1], wl.pad_after[1])
    assert sizes == (wl.N, wl.C_out, OH, OW)
    ref = torch.empty(sizes, device="meta")
    if wl.channels_last:
        ref = ref.contiguous(memory_format=torch.channels_last)
    assert strides == tuple(ref.stride())


def test_known_output_sizes():
    # The five workloads' output planes, by the window-start count.
    got = {}
    for name, wl in WORKLOADS.items():
        got[name] = (oracle.out_size(wl.H, wl.KH, wl.stride[0], wl.pad_before[0], wl.pad_after[0]),
                     wl.C_out)
    assert got["mbv2_dw3x3_s2_bf16_cl"] == (28, 144)
    assert got["grp4x8_9x9_s2_bf16_cl"] == (64, 512)
    assert got["dw4x4_m4_f16_nchw"] == (112, 256)
    assert got["dw7x7_bf16_cl"] == (56, 96)


# ------------------------------------------------------- schedule selection

def test_force_schedule_rules():
    d = bind(x=((1, 8, 8, 8), None), w=((8, 2, 3, 3), None), groups=4)   # grouped, Cin_g 2
    assert gc.conv_select_schedule(d, FAKE, FAKE, None, FAKE) in gc.SCHEDULES
    d.schedule = gc.SCHEDULES["dw_flat"]
    assert gc.conv_select_schedule(d, FAKE, FAKE, None, FAKE) == "dw_flat"
    d.schedule = 17
    assert status_of(lambda: gc.conv_select_schedule(d, FAKE, FAKE, None, FAKE)) == ERR["SCHEDULE"]
    d.schedule = gc.SCHEDULES["dw_row8"]      # depthwise-only schedule on a grouped call
    assert status_of(lambda: gc.conv_select_schedule(d, FAKE, FAKE, None, FAKE)) == ERR["SCHEDULE"]
    assert status_of(lambda: gc.conv_force_schedule(len(gc.SCHEDULES) - 1)) == ERR["SCHEDULE"]
    gc.conv_force_schedule("dw_flat")
    d.schedule = -1
    assert gc.conv_select_schedule(d, FAKE, FAKE, None, FAKE) == "dw_flat"
    gc.conv_force_schedule("auto")


def test_picker_on_the_benchmark_workloads():
    # The picker's schedule for every benchmark workload at full size: the
    # small NCHW depthwise layer runs in one pass (dw_small); the larger ones
    # keep their staged schedules.
    want = {"dw3x3_f32_nchw": "dw_small", "mbv2_dw3x3_s1_bf16_cl": "dw_row8",
            "mbv2_dw3x3_s2_bf16_cl": "dw_row8", "dw7x7_bf16_cl": "dw_row8",
            "dw4x4_m4_f16_nchw": "dw_tc", "grp4x8_9x9_s2_bf16_cl": "grp_tc"}
    for name, sched in want.items():
        wl = WORKLOADS[name]
        xs = cl_strides(wl.N, wl.C_in, wl.H, wl.W) if wl.channels_last else None
        d = bind(x=((wl.N, wl.C_in, wl.H, wl.W), xs),
                 w=((wl.C_out, wl.C_in // wl.groups, wl.KH, wl.KW), None),
                 b=((wl.C_out,), None) if wl.bias else None, stride=tuple(wl.stride),
                 pb=tuple(wl.pad_before), pa=tuple(wl.pad_after), dil=tuple(wl.dilation),
                 groups=wl.groups, dtype=wl.torch_dtype.__str__().split(".")[1])
        got = gc.conv_select_schedule(d, FAKE, FAKE, FAKE if wl.bias else None, FAKE)
        assert got == sched, (name, got)


def test_dw_small_takes_depthwise_only():
    d = bind(x=((2, 8, 9, 11), None), w=((24, 1, 3, 3), None), groups=8)   # multiplier 3
    assert gc.conv_select_schedule(d, FAKE, FAKE, None, FAKE) == "dw_small"
    d.schedule = gc.SCHEDULES["dw_small"]
    assert gc.conv_select_schedule(d, FAKE, FAKE, None, FAKE) == "dw_small"
    d = bind(x=((1, 8, 8, 8), None), w=((8, 2, 3, 3), None), groups=4)     # Cin_g 2
    d.schedule = gc.SCHEDULES["dw_small"]
    assert status_of(lambda: gc.conv_select_schedule(d, FAKE, FAKE, None, FAKE)) == ERR["SCHEDULE"]


def test_dw_tcl_support_rules():
    """dw_tcl takes channels-last 16-bit depthwise calls (multiplier 1) at
    stride 1 and dilation 1 with channels in groups of 8, and nothing else;
    a misaligned input is an alignment error, not a silent fallback."""
    def cl(N, C, H, W, K=3, groups=None, dtype="bfloat16", stride=1, dil=1, cout=None, pad=1):
        cout = cout or C
        return bind(x=((N, C, H, W), cl_strides(N, C, H, W)),
                    w=((cout, C // (groups or C), K, K), None), groups=groups or C,
                    stride=stride, pb=pad, dil=dil, dtype=dtype)

    def forced(d, x=FAKE):
        d.schedule = gc.SCHEDULES["dw_tcl"]
        return status_of(lambda: gc.conv_select_schedule(d, x, FAKE, None, FAKE))

    for dtype in ("bfloat16", "float16"):
        for K in (1, 3, 7, 9):
            assert forced(cl(2, 96, 56, 56, K=K, pad=K // 2, dtype=dtype)) == 0, (dtype, K)
    assert forced(cl(1, 8, 300, 9, K=9, pad=4)) == 0           # taller than a 128-row tile
    assert forced(cl(1, 1232, 9, 12)) == 0                      # more channel groups than SMs
    refused = [
        cl(2, 96, 56, 56, dtype="float32"),                     # fp32
        cl(2, 12, 20, 20),                                      # channels not a multiple of 8
        cl(2, 96, 20, 20, stride=2),                            # stride 2
        cl(2, 96, 20, 20, dil=2, pad=2),                        # dilation 2
        cl(2, 96, 20, 20, cout=192),                            # multiplier 2
        cl(2, 96, 20, 20, groups=48),                           # two channels per group
        bind(x=((2, 96, 20, 20), None), w=((96, 1, 3, 3), None), groups=96,
             dtype="bfloat16"),                                 # NCHW
    ]
    for d in refused:
        assert forced(d) == ERR["SCHEDULE"], (d.C_in, d.stride[0], d.dilation[0], d.layout)
    assert forced(cl(2, 96, 20, 20), x=FAKE + 2) == ERR["ALIGN"]
    # the picker: dw_row8 keeps its square 3/5/7 kernels (the benchmark's
    # 7x7 layer among them); other 2-D kernels of >= 12 taps at stride 1 go
    # to dw_tcl, while small kernels, fp32, dilated and 1-D calls stay on
    # dw_line
    pick = lambda d: gc.conv_select_schedule(d, FAKE, FAKE, None, FAKE)
    assert pick(cl(128, 96, 56, 56, K=7, pad=3)) == "dw_row8"
    assert pick(cl(8, 64, 20, 20)) == "dw_row8"
    for K in (4, 6, 8, 9):
        assert pick(cl(8, 64, 20, 20, K=K, pad=K // 2)) == "dw_tcl", K
    for K in (1, 2):
        assert pick(cl(8, 64, 20, 20, K=K, pad=K // 2)) == "dw_line", K
    nonsquare = bind(x=((8, 64, 20, 20), cl_strides(8, 64, 20, 20)), w=((64, 1, 5, 3), None),
                     groups=64, pb=(2, 1), dtype="float16")
    assert pick(nonsquare) == "dw_tcl"
    assert pick(cl(8, 64, 20, 20, K=4, pad=2, dtype="float32")) == "dw_line"
    assert pick(cl(8, 64, 20, 20, K=4, pad=3, dil=2)) == "dw_line"
    d1 = gc.conv1d_bind(((4, 256, 1000), (1000 * 256, 1, 256)), ((256, 1, 4), (4, 4, 1)), None,
                        1, 3, 0, 1, 256, dtype="bfloat16")
    assert pick(d1) == "dw_line"


def test_dw_forward_refuses_grouped():
    d = bind(x=((1, 8, 8, 8), None), w=((8, 2, 3, 3), None), groups=4)
    assert status_of(lambda: gc.conv_dw_forward(d, FAKE, FAKE, None, FAKE, 0)) == ERR["UNSUPPORTED"]


def test_bias_presence_must_match():
    d = bind()
    assert status_of(lambda: gc.conv_dw_forward(d, FAKE, FAKE, FAKE, FAKE, 0)) == ERR["NULL"]
    d = bind(b=((4,), None))
    assert status_of(lambda: gc.conv_dw_forward(d, FAKE, FAKE, None, FAKE, 0)) == ERR["NULL"]
    assert status_of(lambda: gc.conv_dw_forward(d, None, FAKE, FAKE, FAKE, 0)) == ERR["NULL"]


def test_empty_problem_launches_nothing():
    d = bind(x=((0, 4, 8, 8), None))
    before = gc.conv_launch_count()
    gc.conv_dw_forward(d, FAKE, FAKE, None, FAKE, 0)       # N == 0: OK, no CUDA call
    d = bind(x=((2, 4, 8, 8), None), w=((0, 1, 3, 3), None), groups=4)
    gc.conv_grouped_forward(d, FAKE, FAKE, None, FAKE, 0)  # C_out == 0
    assert gc.conv_launch_count() == before


def test_injected_launch_error_is_reported_without_a_launch():
    d = bind()
    before = gc.conv_launch_count()
    gc.conv_test_inject_launch_error(700)
    assert status_of(lambda: gc.conv_dw_forward(d, FAKE, FAKE, None, FAKE, 0)) == ERR["CUDA"]
    assert gc.conv_last_cuda_error() == 700
    assert gc.conv_launch_count() == before
    gc.conv_test_inject_launch_error(0)
