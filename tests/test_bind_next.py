"""Host logic of the wider envelope, on the CPU: 1-D and transposed binding,
the transposed output-size rule (executorch PR #25091, description, second
paragraph), the dx geometry, schedule selection for dilated / 1-D /
transposed calls (including the stride-1 transposed call that runs as a
flipped-kernel forward), the backward workspace contract and the
desc-kind errors.  No kernel is launched: pointers are fake, aligned device
addresses that are only inspected."""

import ctypes

import pytest
import torch
import torch.nn.functional as F

import grouped_convolution_gb300 as gc
import oracle

ERR = {"NULL": 1, "RANK": 2, "SHAPE": 4, "UNSUPPORTED": 5, "PADDING": 6, "ALIGN": 7, "SCHEDULE": 11,
       "KIND": 12, "WORKSPACE": 13}
FAKE = 1 << 20


@pytest.fixture(scope="module", autouse=True)
def lib():
    gc.build()
    yield
    gc.conv_force_schedule("auto")


def dense(shape):
    strides, acc = [], 1
    for n in reversed(shape):
        strides.insert(0, acc)
        acc *= max(n, 1)
    return (tuple(shape), tuple(strides))


def nlc(N, C, L):
    return ((N, C, L), (L * C, 1, C))


def cl4(N, C, H, W):
    return ((N, C, H, W), (H * W * C, 1, W * C, C))


def status_of(fn):
    try:
        fn()
    except gc.GconvError as e:
        return e.status
    return 0


# ----------------------------------------------------------------------- 1-D

@pytest.mark.parametrize("L,K,s,pb,pa,d", [(100, 4, 1, 3, 0, 1), (77, 7, 2, 3, 3, 1),
                                           (65, 3, 1, 4, 4, 4), (9, 9, 1, 0, 8, 1)])
def test_conv1d_bind_shape_and_layouts(L, K, s, pb, pa, d):
    for xg, want_stride in ((dense((2, 8, L)), None), (nlc(2, 8, L), "nlc")):
        desc = gc.conv1d_bind(xg, dense((8, 1, K)), None, s, pb, pa, d, 8, dtype="bfloat16")
        assert desc.spatial_dims == 1 and desc.H == 1 and desc.KH == 1 and desc.OH == 1
        sizes, strides = gc.out_shape_and_stride(desc)
        OL = oracle.out_size(L, K, s, pb, pa, d)
        assert sizes == (2, 8, OL)
        if want_stride == "nlc":
            assert strides == (OL * 8, 1, 8)
        else:
            assert strides == (8 * OL, OL, 1)
        if pb == pa:
            yt = F.conv1d(torch.zeros(2, 8, L), torch.zeros(8, 1, K), stride=s, padding=pb,
                          dilation=d, groups=8)
            assert tuple(yt.shape) == sizes


def test_conv1d_bind_unbatched_and_rank_errors():
    desc = gc.conv1d_bind(((4, 30), (1, 4)), dense((4, 1, 3)), None, 1, 1, 1, 1, 4,
                          dtype="float32")
    assert desc.unbatched == 1
    sizes, strides = gc.out_shape_and_stride(desc)
    assert sizes == (4, 30) and strides == (1, 4)
    assert status_of(lambda: gc.conv1d_bind(dense((1, 4, 5, 30)), dense((4, 1, 3)), None,
                                            dtype="float32", groups=4)) == ERR["RANK"]
    assert status_of(lambda: gc.conv1d_bind(dense((1, 4, 30)), dense((4, 1, 1, 3)), None,
                                            dtype="float32", groups=4)) == ERR["RANK"]


# ---------------------------------------------------------------- transposed

@pytest.mark.parametrize("H,K,s,p,op,d", [(9, 4, 2, 1, 0, 1), (8, 3, 2, 1, 1, 1),
                                          (10, 3, 1, 1, 0, 1), (7, 3, 3, 0, 2, 2),
                                          (5, 5, 1, 2, 0, 1)])
def test_transpose_bind_matches_torch_shapes(H, K, s, p, op, d):
    desc = gc.conv_transpose_bind(dense((2, 6, H, H + 1)), dense((6, 2, K, K)), None, s, p, p,
                                  op, d, 3, dtype="float32")
    sizes, strides = gc.out_shape_and_stride(desc)
    yt = F.conv_transpose2d(torch.zeros(2, 6, H, H + 1), torch.zeros(6, 2, K, K), stride=s,
                            padding=p, output_padding=op, dilation=d, groups=3)
    assert sizes == tuple(yt.shape)
    assert desc.transposed == 1 and desc.C_out == 6 and desc.Cin_g == 2 and desc.Cout_g == 2
    assert sizes[2] == oracle.transposed_out_size(H, K, s, p, p, op, d)


def test_transpose_bind_asymmetric_crop_and_errors():
    desc = gc.conv_transpose_bind(cl4(1, 16, 5, 7), dense((16, 1, 3, 3)), None, 2, (2, 0),
                                  (0, 3), (1, 0), 1, 16, dtype="bfloat16")
    assert (desc.OH, desc.OW) == ((5 - 1) * 2 + 3 + 1 - 2, (7 - 1) * 2 + 3 - 3)
    assert desc.layout == 1
    # weight's first dim must be C_in
    assert status_of(lambda: gc.conv_transpose_bind(dense((1, 16, 5, 5)), dense((8, 1, 3, 3)),
                                                    None, groups=16, dtype="float32")) \
        == ERR["SHAPE"]
    # crop removes everything
    assert status_of(lambda: gc.conv_transpose_bind(dense((1, 4, 2, 2)), dense((4, 1, 3, 3)),
                                                    None, 1, 2, 2, 0, 1, 4,
                                                    dtype="float32")) == ERR["PADDING"]
    # more than 8 input channels per group
    assert status_of(lambda: gc.conv_transpose_bind(dense((1, 9, 5, 5)), dense((9, 1, 3, 3)),
                                                    None, groups=1, dtype="float32")) \
        == ERR["UNSUPPORTED"]
    d1 = gc.conv_transpose1d_bind(nlc(2, 8, 70), dense((8, 1, 4)), None, 2, 1, 1, 0, 1, 8,
                                  dtype="bfloat16")
    assert gc.out_shape_and_stride(d1) == ((2, 8, 140), (140 * 8, 1, 8))


# ---------------------------------------------------------------- scheduling

def select(desc, aligned=True):
    a = FAKE if aligned else FAKE + 2
    return gc.conv_select_schedule(desc, a, FAKE, None, FAKE)


def test_schedule_selection_wider_envelope():
    # dilation 2, 3x3, stride 1, channels-last depthwise -> dw_row8 (its
    # dilated ring); other dilated channels-last depthwise -> dw_line; a
    # small NCHW dilated one -> dw_small (one pass, any dilation)
    d = gc.conv_bind(cl4(8, 64, 20, 20), dense((64, 1, 3, 3)), None, 1, 2, 2, 2, 64,
                     dtype="bfloat16")
    assert select(d) == "dw_row8"
    for st, dl in ((2, 2), (1, 3)):
        d = gc.conv_bind(cl4(8, 64, 20, 20), dense((64, 1, 3, 3)), None, st, dl, dl, dl, 64,
                         dtype="bfloat16")
        assert select(d) == "dw_line"
        d.schedule = gc.SCHEDULES["dw_row8"]
        assert status_of(lambda: select(d)) == ERR["SCHEDULE"]
    d = gc.conv_bind(cl4(8, 64, 20, 20), dense((64, 1, 5, 5)), None, 1, 4, 4, 2, 64,
                     dtype="bfloat16")
    assert select(d) == "dw_line"
    d = gc.conv_bind(dense((8, 64, 20, 20)), dense((64, 1, 3, 3)), None, 1, 2, 2, 2, 64,
                     dtype="bfloat16")
    assert select(d) == "dw_small"
    for s in ("dw_row8", "dw_mult", "grp_plane", "grp_tc", "dw_tc", "dw_tcl"):
        d.schedule = gc.SCHEDULES[s]
        assert status_of(lambda: select(d)) == ERR["SCHEDULE"]
    # 1-D channels-last depthwise -> dw_line
    d = gc.conv1d_bind(nlc(4, 256, 1000), dense((256, 1, 4)), None, 1, 3, 0, 1, 256,
                       dtype="bfloat16")
    assert select(d) == "dw_line"
    # stride-1 transposed depthwise, channels-last 3x3: a flipped forward on dw_row8
    d = gc.conv_transpose_bind(cl4(8, 64, 20, 20), dense((64, 1, 3, 3)), None, 1, 1, 1, 0, 1,
                               64, dtype="bfloat16")
    assert select(d) == "dw_row8"
    # crop larger than the kernel extent: no flipped form, the transposed gather
    d = gc.conv_transpose_bind(cl4(8, 64, 20, 20), dense((64, 1, 3, 3)), None, 1, 3, 0, 0, 1,
                               64, dtype="bfloat16")
    assert select(d) == "dw_line"
    # stride 2: the transposed gather
    d = gc.conv_transpose_bind(cl4(8, 64, 20, 20), dense((64, 1, 4, 4)), None, 2, 1, 1, 0, 1,
                               64, dtype="bfloat16")
    assert select(d) == "dw_line"
    d.schedule = gc.SCHEDULES["dw_row8"]
    assert status_of(lambda: select(d)) == ERR["SCHEDULE"]
    # stride 2 with a square 3/5/7 kernel: dw_row8's transposed ring (TMA
    # needs a 16-byte aligned input)
    for k in (3, 5, 7):
        d = gc.conv_transpose_bind(cl4(8, 64, 20, 20), dense((64, 1, k, k)), None, 2, k // 2,
                                   k // 2, 1, 1, 64, dtype="bfloat16")
        assert select(d) == "dw_row8"
        assert select(d, aligned=False) != "dw_row8"
        d.schedule = gc.SCHEDULES["dw_row8"]
        assert status_of(lambda: select(d, aligned=False)) == ERR["ALIGN"]
    # ... but not at stride 3, with dilation, or in NCHW
    d = gc.conv_transpose_bind(cl4(8, 64, 20, 20), dense((64, 1, 3, 3)), None, 3, 1, 1, 0, 1,
                               64, dtype="bfloat16")
    assert select(d) == "dw_line"
    d = gc.conv_transpose_bind(cl4(8, 64, 20, 20), dense((64, 1, 3, 3)), None, 2, 2, 2, 1, 2,
                               64, dtype="bfloat16")
    assert select(d) == "dw_line"
    d = gc.conv_transpose_bind(dense((8, 64, 20, 20)), dense((64, 1, 3, 3)), None, 2, 1, 1, 1, 1,
                               64, dtype="bfloat16")
    assert select(d) != "dw_row8"


def test_kind_errors_and_dx_geometry():
    lib = gc._load()
    fwd = gc.conv_bind(cl4(2, 16, 9, 9), dense((16, 1, 3, 3)), None, 2, 1, 1, 1, 16,
                       dtype="bfloat16")
    tr = gc.conv_transpose_bind(cl4(2, 16, 9, 9), dense((16, 1, 3, 3)), None, 2, 1, 1, 0, 1,
                                16, dtype="bfloat16")
    assert lib.conv_transpose_forward(ctypes.byref(fwd), FAKE, FAKE, None, FAKE, None) \
        == ERR["KIND"]
    assert lib.conv_grouped_forward(ctypes.byref(tr), FAKE, FAKE, None, FAKE, None) \
        == ERR["KIND"]
    assert lib.conv_dw_forward(ctypes.byref(tr), FAKE, FAKE, None, FAKE, None) == ERR["KIND"]
    assert lib.conv_backward_input(ctypes.byref(tr), FAKE, FAKE, FAKE, None) == ERR["KIND"]
    assert status_of(lambda: gc.grad_input_shape_and_stride(tr)) == ERR["KIND"]
    sizes, strides = gc.grad_input_shape_and_stride(fwd)
    assert sizes == (2, 16, 9, 9) and strides == (9 * 9 * 16, 1, 9 * 16, 16)
    d1 = gc.conv1d_bind(((16, 50), (50, 1)), dense((16, 1, 3)), None, 1, 1, 1, 1, 16,
                        dtype="float32")
    assert gc.grad_input_shape_and_stride(d1) == ((16, 50), (50, 1))


def test_backward_weight_workspace_contract():
    lib = gc._load()
    d = gc.conv_bind(cl4(32, 144, 56, 56), dense((144, 1, 3, 3)), None, 1, 1, 1, 1, 144,
                     dtype="bfloat16")
    need = gc.conv_backward_weight_workspace_size(d)
    assert need >= 144 * 10 * 4 and need % 4 == 0
    assert need == gc.conv_backward_weight_workspace_size(d)   # a function of the shape
    # missing, short or misaligned workspace: refused before any launch
    for ws, nbytes in ((None, need), (FAKE, need - 4), (FAKE + 4, need)):
        assert lib.conv_backward_weight(ctypes.byref(d), FAKE, FAKE, FAKE, None, ws, nbytes,
                                        None) == ERR["WORKSPACE"]
    assert lib.conv_backward_weight(ctypes.byref(d), FAKE, FAKE, None, None, FAKE, need,
                                    None) == ERR["NULL"]
    tr = gc.conv_transpose_bind(cl4(2, 16, 9, 9), dense((16, 1, 3, 3)), None, 2, 1, 1, 0, 1,
                                16, dtype="bfloat16")
    assert status_of(lambda: gc.conv_backward_weight_workspace_size(tr)) == ERR["KIND"]


def test_backward_weight_workspace_covers_the_row_ring():
    # Channels-last depthwise square 3/5/7 kernels at stride 1 or 2 take the
    # row-ring partial pass: one fp32 slice of C_out x (KH*KW + 1) per
    # persistent CTA (two per SM for 3x3, one for 5x5 / 7x7, 152 SMs).
    for C, H, K, s in ((144, 56, 3, 1), (144, 56, 3, 2), (96, 56, 7, 1), (24, 112, 5, 2)):
        d = gc.conv_bind(cl4(32, C, H, H), dense((C, 1, K, K)), None, s, K // 2, K // 2, 1, C,
                         dtype="bfloat16")
        per_sm = 2 if K == 3 else 1
        assert gc.conv_backward_weight_workspace_size(d) >= 152 * per_sm * C * (K * K + 1) * 4


def test_injected_error_on_new_entry_points():
    lib = gc._load()
    tr = gc.conv_transpose_bind(cl4(2, 16, 9, 9), dense((16, 1, 3, 3)), None, 2, 1, 1, 0, 1,
                                16, dtype="bfloat16")
    gc.conv_test_inject_launch_error(700)
    assert lib.conv_transpose_forward(ctypes.byref(tr), FAKE, FAKE, None, FAKE, None) == 8
    assert gc.conv_last_cuda_error() == 700
    fwd = gc.conv_bind(cl4(2, 16, 9, 9), dense((16, 1, 3, 3)), None, 1, 1, 1, 1, 16,
                       dtype="bfloat16")
    need = gc.conv_backward_weight_workspace_size(fwd)
    gc.conv_test_inject_launch_error(701)
    assert lib.conv_backward_weight(ctypes.byref(fwd), FAKE, FAKE, FAKE, FAKE, FAKE, need,
                                    None) == 8
    gc.conv_test_inject_launch_error(702)
    assert lib.conv_backward_input(ctypes.byref(fwd), FAKE, FAKE, FAKE, None) == 8
    assert gc.conv_last_cuda_error() == 702
    # the fixed-buffer weight gradient: size check first, then the hook
    assert need <= gc.conv_backward_weight_noalloc_limit()
    gc.conv_test_inject_launch_error(703)
    assert lib.conv_backward_weight_noalloc(ctypes.byref(fwd), FAKE, FAKE, FAKE, FAKE,
                                            None) == 8
    assert gc.conv_last_cuda_error() == 703
    gc.conv_test_inject_launch_error(0)
