"""Pins for the oracle's dilated, 1-D, transposed and backward functions (no GPU).

Each function is checked against something other than itself:
  - dilated forward: an independent brute-force im2col whose windows take
    every d-th input, the zero-inserted-kernel identity (a dilated kernel is
    the undilated kernel with d-1 zeros between its taps), the window-start
    enumeration for the output size and torch's CPU float64 conv2d;
  - 1-D: torch's CPU float64 conv1d (after an explicit pad for asymmetric
    padding) and the 2-D brute force on a height-1 image;
  - transposed (executorch PR #25091 "Run transposed convolutions on the
    implicit-GEMM template", description, second paragraph: output o reads,
    at tap k, input (o + padding_before - k) / stride when that is an
    integer inside the input; the [C_in, C_out/groups, ...] weight): an
    independent scatter (every input adds w * x at i*s + k*d of an uncropped
    output that is then cropped), the adjoint identity with the pinned
    forward oracle (<conv(x), y> = <x, conv_transpose(y)>), zero-insertion
    upsampling for a 1x1 unit kernel, and torch's CPU float64
    conv_transpose2d / conv_transpose1d;
  - backward (the gradients torch/_inductor/kernel/conv.py,
    convolution_backward_lowering, produces): the adjoint identities
    <conv(x; w), gy> = <x, dx> = <w, dw>, db = the sum of gy, the transposed
    oracle with the geometry that maps the output back onto the input, and
    torch's CPU float64 autograd.
"""


import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ dilation

def im2col_dilated(x, w, b, stride, pb, pa, groups, dil):
    """Brute force: pad explicitly, gather each window's taps d apart into a
    row, multiply by the per-group weight matrix."""
    N, C, H, W = x.shape
    Co, Cig, KH, KW = w.shape
    sh, sw = stride
    dh, dw = dil
    xp = np.pad(x, ((0, 0), (0, 0), (pb[0], pa[0]), (pb[1], pa[1])))
    Hp, Wp = xp.shape[2:]
    eh, ew = dh * (KH - 1) + 1, dw * (KW - 1) + 1
    starts_h = list(range(0, Hp - eh + 1, sh))
    starts_w = list(range(0, Wp - ew + 1, sw))
    Cog = Co // groups
    y = np.zeros((N, Co, len(starts_h), len(starts_w)))
    yabs = np.zeros_like(y)
    for g in range(groups):
        xg = xp[:, g * Cig:(g + 1) * Cig]
        Wg = w[g * Cog:(g + 1) * Cog].reshape(Cog, -1)
        for i, th in enumerate(starts_h):
            for j, tw in enumerate(starts_w):
                win = xg[:, :, th:th + eh:dh, tw:tw + ew:dw].reshape(N, -1)
                y[:, g * Cog:(g + 1) * Cog, i, j] = win @ Wg.T
                yabs[:, g * Cog:(g + 1) * Cog, i, j] = np.abs(win) @ np.abs(Wg).T
    if b is not None:
        y += b[None, :, None, None]
    return y, yabs


DIL_CASES = [
    # (N, Cig, Cog, G, H, W, KH, KW, stride, pb, pa, dil)
    (1, 1, 1, 3, 9, 9, 3, 3, (1, 1), (2, 2), (2, 2), (2, 2)),
    (2, 1, 2, 2, 11, 8, 3, 2, (2, 1), (3, 1), (1, 2), (3, 2)),
    (1, 4, 8, 2, 10, 10, 3, 3, (1, 2), (0, 2), (4, 0), (2, 3)),
    (1, 2, 1, 3, 7, 13, 1, 5, (1, 1), (0, 4), (0, 4), (1, 2)),
    (1, 1, 4, 2, 12, 12, 4, 4, (3, 3), (3, 3), (3, 3), (2, 2)),
    (1, 8, 1, 1, 9, 9, 2, 2, (1, 1), (0, 0), (0, 0), (8, 8)),   # span = whole input
]


@pytest.mark.parametrize("case", DIL_CASES)
def test_dilated_matches_brute_force(case):
    N, Cig, Cog, G, H, W, KH, KW, s, pb, pa, d = case
    r = rng(hash(case) % 997)
    x = r.standard_normal((N, Cig * G, H, W))
    w = r.standard_normal((Cog * G, Cig, KH, KW))
    b = r.standard_normal(Cog * G)
    y, bound = oracle.conv2d(x, w, b, s, pb, pa, G, d)
    y_ref, abs_ref = im2col_dilated(x, w, b, s, pb, pa, G, d)
    assert y.shape == y_ref.shape
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(bound, abs_ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("case", DIL_CASES)
def test_dilated_equals_zero_inserted_kernel(case):
    N, Cig, Cog, G, H, W, KH, KW, s, pb, pa, d = case
    r = rng(hash(case) % 991)
    x = r.standard_normal((N, Cig * G, H, W))
    w = r.standard_normal((Cog * G, Cig, KH, KW))
    wz = np.zeros((Cog * G, Cig, d[0] * (KH - 1) + 1, d[1] * (KW - 1) + 1))
    wz[:, :, ::d[0], ::d[1]] = w
    y, _ = oracle.conv2d(x, w, None, s, pb, pa, G, d)
    yz, _ = oracle.conv2d(x, wz, None, s, pb, pa, G, 1)
    np.testing.assert_allclose(y, yz, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("case", DIL_CASES)
def test_dilated_matches_torch_cpu_f64(case):
    N, Cig, Cog, G, H, W, KH, KW, s, pb, pa, d = case
    r = rng(hash(case) % 983)
    x = r.standard_normal((N, Cig * G, H, W))
    w = r.standard_normal((Cog * G, Cig, KH, KW))
    b = r.standard_normal(Cog * G)
    y, _ = oracle.conv2d(x, w, b, s, pb, pa, G, d)
    xt = F.pad(torch.from_numpy(x), (pb[1], pa[1], pb[0], pa[0]))
    yt = F.conv2d(xt, torch.from_numpy(w), torch.from_numpy(b), stride=s, dilation=d,
                  groups=G)
    np.testing.assert_allclose(y, yt.numpy(), rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("H,K,s,pb,pa,d", [
    (10, 3, 1, 0, 0, 2), (10, 3, 2, 1, 2, 3), (5, 3, 1, 0, 0, 2), (4, 3, 1, 0, 0, 2),
    (9, 9, 1, 4, 4, 2), (1, 2, 1, 0, 0, 5), (7, 4, 3, 2, 0, 2)])
def test_dilated_out_size(H, K, s, pb, pa, d):
    span = d * (K - 1) + 1
    starts = [t for t in range(0, H + pb + pa) if t % s == 0 and t + span <= H + pb + pa]
    got = oracle.out_size(H, K, s, pb, pa, d)
    assert got == (len(starts) if starts else -1)
    if starts:
        # ATen's formula for symmetric padding folds (pb + pa) in the same way
        assert got == (H + pb + pa - span) // s + 1


# ----------------------------------------------------------------------- 1-D

@pytest.mark.parametrize("N,C,L,m,K,s,pb,pa,d", [
    (2, 6, 37, 1, 4, 1, 3, 0, 1),      # causal depthwise, kernel 4
    (1, 4, 50, 2, 7, 2, 3, 3, 1),
    (3, 8, 29, 1, 3, 1, 2, 2, 2),
    (1, 2, 9, 3, 9, 1, 0, 8, 1),
])
def test_conv1d_matches_torch_cpu_f64(N, C, L, m, K, s, pb, pa, d):
    r = rng(N * 100 + L)
    x = r.standard_normal((N, C, L))
    w = r.standard_normal((C * m, 1, K))
    b = r.standard_normal(C * m)
    y, bound = oracle.conv1d(x, w, b, s, pb, pa, C, d)
    yt = F.conv1d(F.pad(torch.from_numpy(x), (pb, pa)), torch.from_numpy(w),
                  torch.from_numpy(b), stride=s, dilation=d, groups=C)
    np.testing.assert_allclose(y, yt.numpy(), rtol=1e-11, atol=1e-11)
    y2, b2 = im2col_dilated(x[:, :, None, :], w[:, :, None, :], b, (1, s), (0, pb),
                            (0, pa), C, (1, d))
    np.testing.assert_allclose(bound, b2[:, :, 0, :], rtol=1e-12, atol=1e-12)


def test_conv1d_unbatched():
    r = rng(5)
    x = r.standard_normal((4, 20))
    w = r.standard_normal((4, 1, 3))
    y, _ = oracle.conv1d(x, w, None, 1, 1, 1, 4)
    y1, _ = oracle.conv1d(x[None], w, None, 1, 1, 1, 4)
    np.testing.assert_array_equal(y, y1)


# ---------------------------------------------------------------- transposed

def scatter_transposed(x, w, b, stride, pb, pa, op, groups, dil):
    """Independent scatter: every input pixel adds w * x at i*s + k*d of an
    uncropped output (extended by output_padding at the end), which is then
    cropped by pb before and pa after."""
    N, C_in, H, W = x.shape
    _, Cog, KH, KW = w.shape
    sh, sw = stride
    dh, dw = dil
    Cig = C_in // groups
    Co = Cog * groups
    FH = (H - 1) * sh + dh * (KH - 1) + 1 + op[0]
    FW = (W - 1) * sw + dw * (KW - 1) + 1 + op[1]
    full = np.zeros((N, Co, FH, FW))
    fabs_ = np.zeros_like(full)
    for c in range(C_in):
        g = c // Cig
        for j in range(Cog):
            co = g * Cog + j
            for kh in range(KH):
                for kw in range(KW):
                    p = w[c, j, kh, kw] * x[:, c]
                    hs = slice(kh * dh, kh * dh + (H - 1) * sh + 1, sh)
                    ws = slice(kw * dw, kw * dw + (W - 1) * sw + 1, sw)
                    full[:, co, hs, ws] += p
                    fabs_[:, co, hs, ws] += np.abs(p)
    y = full[:, :, pb[0]:FH - pa[0], pb[1]:FW - pa[1]]
    yabs = fabs_[:, :, pb[0]:FH - pa[0], pb[1]:FW - pa[1]]
    if b is not None:
        y = y + b[None, :, None, None]
    return y, yabs


T_CASES = [
    # (N, Cig, Cog, G, H, W, KH, KW, stride, pb, pa, op, dil)
    (1, 1, 1, 3, 5, 6, 4, 4, (2, 2), (1, 1), (1, 1), (0, 0), (1, 1)),    # 2x upsampling
    (2, 1, 2, 2, 4, 5, 3, 3, (2, 2), (1, 1), (1, 1), (1, 1), (1, 1)),    # output_padding
    (1, 4, 2, 2, 5, 4, 3, 5, (1, 3), (2, 0), (0, 3), (0, 2), (1, 1)),    # asymmetric crop
    (1, 2, 3, 1, 4, 4, 3, 3, (3, 2), (0, 0), (0, 0), (2, 0), (2, 1)),    # dilated
    (1, 8, 1, 1, 3, 3, 9, 9, (1, 1), (4, 4), (4, 4), (0, 0), (1, 1)),
    (1, 1, 4, 2, 6, 3, 1, 1, (3, 3), (0, 0), (0, 0), (0, 0), (1, 1)),    # 1x1 strided
    (2, 3, 1, 2, 1, 7, 2, 4, (2, 1), (1, 0), (0, 2), (1, 0), (1, 2)),
]


@pytest.mark.parametrize("case", T_CASES)
@pytest.mark.parametrize("bias", [False, True])
def test_transposed_matches_scatter(case, bias):
    N, Cig, Cog, G, H, W, KH, KW, s, pb, pa, op, d = case
    r = rng(hash(case) % 977 + bias)
    x = r.standard_normal((N, Cig * G, H, W))
    w = r.standard_normal((Cig * G, Cog, KH, KW))
    b = r.standard_normal(Cog * G) if bias else None
    y, bound = oracle.conv_transpose2d(x, w, b, s, pb, pa, op, G, d)
    y_ref, abs_ref = scatter_transposed(x, w, b, s, pb, pa, op, G, d)
    assert y.shape == y_ref.shape
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(bound, abs_ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("case", T_CASES)
def test_transposed_matches_torch_cpu_f64(case):
    N, Cig, Cog, G, H, W, KH, KW, s, pb, pa, op, d = case
    r = rng(hash(case) % 971)
    x = r.standard_normal((N, Cig * G, H, W))
    w = r.standard_normal((Cig * G, Cog, KH, KW))
    b = r.standard_normal(Cog * G)
    y, _ = oracle.conv_transpose2d(x, w, b, s, pb, pa, op, G, d)
    # torch crops symmetrically and bounds output_padding; take its uncropped
    # result (nothing lands past its end, so output_padding appends zeros)
    # and crop it here.
    yt = F.conv_transpose2d(torch.from_numpy(x), torch.from_numpy(w), None,
                            stride=s, groups=G, dilation=d).numpy()
    yt = np.pad(yt, ((0, 0), (0, 0), (0, op[0]), (0, op[1])))
    yt = yt[:, :, pb[0]:yt.shape[2] - pa[0], pb[1]:yt.shape[3] - pa[1]]
    yt = yt + b[None, :, None, None]
    np.testing.assert_allclose(y, yt, rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("case", T_CASES)
def test_transposed_is_adjoint_of_forward(case):
    # <conv(u; w), v> == <u, conv_transpose(v; w)> for u of the transposed
    # output's size and v of its input's size, with the same stride, padding,
    # dilation and groups, and the transposed weight read as the forward
    # weight [C_out_fwd = C_in_t, Cin_g_fwd = Cout_g_t, KH, KW].
    N, Cig, Cog, G, H, W, KH, KW, s, pb, pa, op, d = case
    r = rng(hash(case) % 967)
    v = r.standard_normal((N, Cig * G, H, W))
    w = r.standard_normal((Cig * G, Cog, KH, KW))
    t, _ = oracle.conv_transpose2d(v, w, None, s, pb, pa, op, G, d)
    OH, OW = t.shape[2:]
    u = r.standard_normal((N, Cog * G, OH, OW))
    # the forward conv of u with pad_before pb covers outputs 0..H-1 once
    # enough zeros follow u (pa + op suffices); the rest is cut off.
    pa_f = (pa[0] + op[0], pa[1] + op[1])
    fy, _ = oracle.conv2d(u, w, None, s, pb, pa_f, G, d)
    fy = fy[:, :, :H, :W]
    assert fy.shape == v.shape
    lhs = float(np.sum(fy * v))
    rhs = float(np.sum(u * t))
    assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(lhs))


def test_transposed_unit_kernel_is_zero_insertion():
    r = rng(3)
    x = r.standard_normal((2, 3, 4, 5))
    w = np.ones((3, 1, 1, 1))
    y, _ = oracle.conv_transpose2d(x, w, None, (3, 2), 0, 0, 0, 3)
    expect = np.zeros((2, 3, 10, 9))
    expect[:, :, ::3, ::2] = x
    np.testing.assert_array_equal(y, expect)


@pytest.mark.parametrize("H,K,s,pb,pa,op,d", [
    (5, 4, 2, 1, 1, 0, 1), (4, 3, 2, 1, 1, 1, 1), (3, 9, 1, 4, 4, 0, 1),
    (4, 3, 3, 0, 0, 2, 2), (1, 2, 1, 0, 0, 0, 5), (6, 1, 3, 0, 0, 0, 1)])
def test_transposed_out_size(H, K, s, pb, pa, op, d):
    got = oracle.transposed_out_size(H, K, s, pb, pa, op, d)
    assert got == (H - 1) * s + d * (K - 1) + 1 + op - pb - pa
    if pb == pa and op < max(s, d):
        x = torch.zeros(1, 1, 1, H, dtype=torch.float64)
        w = torch.zeros(1, 1, 1, K, dtype=torch.float64)
        yt = F.conv_transpose2d(x, w, stride=(1, s), padding=(0, pb),
                                output_padding=(0, op), dilation=(1, d))
        assert yt.shape[-1] == got


def test_transposed_out_size_rejects():
    assert oracle.transposed_out_size(3, 3, 1, 3, 3, 0, 1) == -1   # cropped away
    assert oracle.transposed_out_size(0, 3, 1, 0, 0, 0, 1) == -1
    assert oracle.transposed_out_size(3, 3, 1, -1, 0, 0, 1) == -1


@pytest.mark.parametrize("N,C,L,m,K,s,p,op", [
    (2, 4, 16, 1, 4, 2, 1, 0),       # 1-D upsampling, kernel 4 stride 2
    (1, 3, 9, 2, 3, 3, 1, 2),
])
def test_conv_transpose1d_matches_torch(N, C, L, m, K, s, p, op):
    r = rng(L)
    x = r.standard_normal((N, C, L))
    w = r.standard_normal((C, m, K))
    y, _ = oracle.conv_transpose1d(x, w, None, s, p, p, op, C)
    yt = F.conv_transpose1d(torch.from_numpy(x), torch.from_numpy(w), stride=s,
                            padding=p, output_padding=op, groups=C)
    np.testing.assert_allclose(y, yt.numpy(), rtol=1e-11, atol=1e-11)


# ------------------------------------------------------------------ backward

B_CASES = [
    # (N, Cig, Cog, G, H, W, KH, KW, stride, pb, pa, dil)
    (2, 1, 1, 3, 7, 6, 3, 3, (1, 1), (1, 1), (1, 1), (1, 1)),
    (1, 1, 4, 2, 9, 8, 4, 4, (1, 1), (1, 1), (2, 2), (1, 1)),
    (1, 4, 8, 2, 11, 10, 5, 3, (2, 2), (2, 1), (2, 1), (1, 1)),    # grouped, stride 2
    (2, 2, 3, 2, 8, 9, 3, 2, (3, 2), (0, 1), (2, 0), (1, 1)),      # remainder rows
    (1, 1, 1, 4, 10, 10, 3, 3, (1, 2), (2, 2), (2, 2), (2, 2)),    # dilated
    (1, 8, 1, 1, 5, 5, 5, 5, (1, 1), (0, 0), (0, 0), (1, 1)),      # one output pixel ring
]


def _bwd_case(case, seed):
    N, Cig, Cog, G, H, W, KH, KW, s, pb, pa, d = case
    r = rng(seed)
    x = r.standard_normal((N, Cig * G, H, W))
    w = r.standard_normal((Cog * G, Cig, KH, KW))
    y, _ = oracle.conv2d(x, w, None, s, pb, pa, G, d)
    gy = r.standard_normal(y.shape)
    return x, w, y, gy


@pytest.mark.parametrize("case", B_CASES)
def test_backward_adjoint_identities(case):
    N, Cig, Cog, G, H, W, KH, KW, s, pb, pa, d = case
    x, w, y, gy = _bwd_case(case, hash(case) % 953)
    g = oracle.conv2d_backward(x, w, gy, s, pb, pa, G, d)
    dx, dw, db = g["dx"][0], g["dw"][0], g["db"][0]
    inner = float(np.sum(y * gy))           # the forward is bilinear in (x, w)
    assert abs(float(np.sum(x * dx)) - inner) <= 1e-10 * max(1.0, abs(inner))
    assert abs(float(np.sum(w * dw)) - inner) <= 1e-10 * max(1.0, abs(inner))
    np.testing.assert_allclose(db, gy.sum(axis=(0, 2, 3)), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("case", B_CASES)
def test_backward_matches_torch_autograd(case):
    N, Cig, Cog, G, H, W, KH, KW, s, pb, pa, d = case
    x, w, _, gy = _bwd_case(case, hash(case) % 947)
    b = rng(1).standard_normal(Cog * G)
    g = oracle.conv2d_backward(x, w, gy, s, pb, pa, G, d)
    xt = torch.from_numpy(x).requires_grad_()
    wt = torch.from_numpy(w).requires_grad_()
    bt = torch.from_numpy(b).requires_grad_()
    yt = F.conv2d(F.pad(xt, (pb[1], pa[1], pb[0], pa[0])), wt, bt, stride=s, dilation=d,
                  groups=G)
    yt.backward(torch.from_numpy(gy))
    np.testing.assert_allclose(g["dx"][0], xt.grad.numpy(), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(g["dw"][0], wt.grad.numpy(), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(g["db"][0], bt.grad.numpy(), rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("case", B_CASES)
def test_backward_dx_is_transposed_conv(case):
    # dx is the transposed convolution of gy with the forward weight, cropped
    # by pad_before and sized back to H x W (output_padding / crop after).
    N, Cig, Cog, G, H, W, KH, KW, s, pb, pa, d = case
    x, w, _, gy = _bwd_case(case, hash(case) % 941)
    g = oracle.conv2d_backward(x, w, gy, s, pb, pa, G, d, need=("dx",))
    OH, OW = gy.shape[2:]
    pa_t, op_t = [], []
    for L, O, K, ss, p, dd in ((H, OH, KH, s[0], pb[0], d[0]), (W, OW, KW, s[1], pb[1], d[1])):
        full = (O - 1) * ss + dd * (K - 1) + 1
        r = L + p - full
        pa_t.append(max(0, -r))
        op_t.append(max(0, r))
    t, tb = oracle.conv_transpose2d(gy, w, None, s, pb, tuple(pa_t), tuple(op_t), G, d)
    np.testing.assert_allclose(g["dx"][0], t, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dx"][1], tb, rtol=1e-12, atol=1e-12)


def test_backward_bounds_are_abs_sums():
    case = B_CASES[2]
    N, Cig, Cog, G, H, W, KH, KW, s, pb, pa, d = case
    x, w, _, gy = _bwd_case(case, 11)
    g = oracle.conv2d_backward(x, w, gy, s, pb, pa, G, d)
    ga = oracle.conv2d_backward(np.abs(x), np.abs(w), np.abs(gy), s, pb, pa, G, d)
    for k in ("dx", "dw", "db"):
        np.testing.assert_allclose(g[k][1], ga[k][0], rtol=1e-12, atol=1e-12)
        assert np.all(np.abs(g[k][0]) <= g[k][1] * (1 + 1e-12) + 1e-12)


def test_backward_unbatched_and_partial():
    r = rng(2)
    x = r.standard_normal((3, 6, 6))
    w = r.standard_normal((3, 1, 3, 3))
    gy = r.standard_normal((3, 6, 6))
    g = oracle.conv2d_backward(x, w, gy, 1, 1, 1, 3, need=("dw",))
    assert set(g) == {"dw"}
    g1 = oracle.conv2d_backward(x[None], w, gy[None], 1, 1, 1, 3)
    np.testing.assert_array_equal(g["dw"][0], g1["dw"][0])
    g2 = oracle.conv2d_backward(x, w, gy, 1, 1, 1, 3, need=("dx",))
    assert g2["dx"][0].shape == x.shape
