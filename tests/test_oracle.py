"""Pins for the CPU fp64 oracle (no GPU).

The oracle is checked against things other than itself: an independent
brute-force im2col product, hand-derived values, closed forms (delta and
identity kernels, constant inputs), an enumeration of window starts for the
output size, linearity / subsampling / padding / grouping invariants, and, as
a library special case, torch's own CPU float64 convolution.  Each is chosen
so that a dropped term, a wrong sign or index, a swapped operand or a wrong
group mapping in the oracle fails at least one of them.

Semantics pinned (cross-correlation, zero padding, output index o reads input
o*s - pad_before + k at tap k, group g owns input channels [g*Cin_g, ...) and
output channels [g*Cout_g, ...)): torch/_inductor/kernel/conv.py,
LOOP_BODY_2D and conv2d_template; explicit padding_before/padding_after:
executorch PR #25084, description.
"""

import itertools
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def rng(seed):
    return np.random.default_rng(seed)


def im2col_conv(x, w, b, stride, pb, pa, groups):
    """Independent brute force: pad explicitly, unfold every window into a
    row, multiply by the reshaped per-group weight matrix."""
    N, C, H, W = x.shape
    Co, Cig, KH, KW = w.shape
    sh, sw = stride
    xp = np.pad(x, ((0, 0), (0, 0), (pb[0], pa[0]), (pb[1], pa[1])))
    Hp, Wp = xp.shape[2:]
    starts_h = list(range(0, Hp - KH + 1, sh))
    starts_w = list(range(0, Wp - KW + 1, sw))
    OH, OW = len(starts_h), len(starts_w)
    Cog = Co // groups
    y = np.zeros((N, Co, OH, OW))
    yabs = np.zeros((N, Co, OH, OW))
    for g in range(groups):
        xg = xp[:, g * Cig:(g + 1) * Cig]
        cols = np.empty((N, OH, OW, Cig * KH * KW))
        for i, th in enumerate(starts_h):
            for j, tw in enumerate(starts_w):
                cols[:, i, j, :] = xg[:, :, th:th + KH, tw:tw + KW].reshape(N, -1)
        A = cols.reshape(N * OH * OW, -1)
        B = w[g * Cog:(g + 1) * Cog].reshape(Cog, -1).T
        y[:, g * Cog:(g + 1) * Cog] = (A @ B).reshape(N, OH, OW, Cog).transpose(0, 3, 1, 2)
        yabs[:, g * Cog:(g + 1) * Cog] = (np.abs(A) @ np.abs(B)).reshape(
            N, OH, OW, Cog).transpose(0, 3, 1, 2)
    if b is not None:
        y = y + b[None, :, None, None]
    return y, yabs


def random_case(seed, N, Cig, Cog, G, H, W, KH, KW, bias=True):
    r = rng(seed)
    x = r.standard_normal((N, Cig * G, H, W))
    w = r.standard_normal((Cog * G, Cig, KH, KW))
    b = r.standard_normal(Cog * G) if bias else None
    return x, w, b


# ---------------------------------------------------------------- brute force

BRUTE_CASES = [
    # (N, Cig, Cog, G, H, W, KH, KW, stride, pb, pa)
    (1, 1, 1, 3, 5, 5, 3, 3, (1, 1), (1, 1), (1, 1)),        # depthwise
    (2, 1, 4, 2, 7, 6, 4, 4, (1, 1), (1, 1), (2, 2)),        # multiplier 4, 'same' asym
    (1, 1, 2, 3, 9, 9, 9, 9, (2, 2), (4, 4), (4, 4)),        # 9x9 s2
    (1, 4, 8, 2, 8, 8, 3, 5, (2, 1), (1, 2), (0, 3)),        # grouped 4->8, non-square
    (2, 8, 1, 1, 6, 7, 2, 3, (3, 2), (0, 1), (2, 0)),        # Cin_g 8, one output
    (1, 2, 3, 4, 5, 9, 1, 9, (1, 3), (0, 4), (0, 4)),        # 1x9 strip kernel
    (1, 3, 2, 1, 4, 4, 5, 5, (1, 1), (2, 2), (2, 2)),        # window larger than input
    (1, 1, 1, 2, 3, 3, 1, 1, (2, 2), (0, 0), (0, 0)),        # 1x1 strided
    (1, 1, 17, 1, 6, 5, 3, 2, (1, 1), (1, 0), (1, 1)),       # multiplier 17
    (1, 5, 3, 2, 7, 7, 7, 1, (4, 1), (3, 0), (3, 0)),        # stride > kernel width
]


@pytest.mark.parametrize("case", BRUTE_CASES)
@pytest.mark.parametrize("bias", [False, True])
def test_oracle_matches_brute_force_im2col(case, bias):
    N, Cig, Cog, G, H, W, KH, KW, s, pb, pa = case
    x, w, b = random_case(hash(case) % 1000 + bias, N, Cig, Cog, G, H, W, KH, KW, bias)
    y, bound = oracle.conv2d(x, w, b, s, pb, pa, G)
    y_ref, abs_ref = im2col_conv(x, w, b, s, pb, pa, G)
    assert y.shape == y_ref.shape
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(bound, abs_ref, rtol=1e-12, atol=1e-12)


def test_points_equal_full():
    x, w, b = random_case(7, 2, 4, 8, 3, 11, 10, 5, 3)
    y, bound = oracle.conv2d(x, w, b, (2, 1), (2, 1), (1, 2), 3)
    r = rng(8)
    pts = np.stack([r.integers(0, n, 50) for n in y.shape], axis=1)
    yp, bp = oracle.conv2d_points(x, w, b, (2, 1), (2, 1), (1, 2), 3, pts)
    np.testing.assert_array_equal(yp, y[tuple(pts.T)])
    np.testing.assert_array_equal(bp, bound[tuple(pts.T)])


# ------------------------------------------------------------- hand-derived

def test_hand_worked_example():
    # x = [[1,2,3],[4,5,6],[7,8,9]], w = [[1,0],[0,-1]], no padding, stride 1:
    #   y[0,0] = 1*1 - 5 = -4, y[0,1] = 2 - 6 = -4, y[1,0] = 4 - 8 = -4,
    #   y[1,1] = 5 - 9 = -4.  With pad_before=1, pad_after=0 the extra first
    #   row/column see only the -1 tap: y'[0,0] = -1, y'[0,1] = -2, y'[1,0] = -4.
    x = np.arange(1, 10, dtype=np.float64).reshape(1, 1, 3, 3)
    w = np.array([[1.0, 0.0], [0.0, -1.0]]).reshape(1, 1, 2, 2)
    y, _ = oracle.conv2d(x, w, None, 1, 0, 0, 1)
    np.testing.assert_array_equal(y[0, 0], [[-4, -4], [-4, -4]])
    y2, bound2 = oracle.conv2d(x, w, None, 1, (1, 1), (0, 0), 1)
    np.testing.assert_array_equal(y2[0, 0], [[-1, -2, -3], [-4, -4, -4], [-7, -4, -4]])
    # bound at (1,1) of the padded case: |1*1| + |-1*5| = 6
    assert bound2[0, 0, 1, 1] == 6.0
    # stride 2 over the padded 4x4 input: rows/cols starts 0 and 2
    y3, _ = oracle.conv2d(x, w, None, 2, (1, 1), (0, 0), 1)
    np.testing.assert_array_equal(y3[0, 0], [[-1, -3], [-7, -4]])


def test_hand_worked_grouped_mapping():
    # 2 groups, 2 in / 1 out per group, 1x1 kernel: output channel co reads
    # input channels 2*co and 2*co+1 only (group g owns [g*Cin_g, (g+1)*Cin_g)).
    x = np.array([1.0, 10.0, 100.0, 1000.0]).reshape(1, 4, 1, 1)
    w = np.array([[1.0, 2.0], [3.0, 4.0]]).reshape(2, 2, 1, 1)
    y, _ = oracle.conv2d(x, w, np.array([0.5, -0.5]), 1, 0, 0, 2)
    np.testing.assert_array_equal(y.reshape(-1), [1 + 20 + 0.5, 300 + 4000 - 0.5])


def test_hand_worked_multiplier_mapping():
    # depthwise multiplier 2: output channel c*m + j reads input channel c.
    x = np.array([2.0, 3.0]).reshape(1, 2, 1, 1)
    w = np.array([1.0, 10.0, 100.0, 1000.0]).reshape(4, 1, 1, 1)
    y, _ = oracle.conv2d(x, w, None, 1, 0, 0, 2)
    np.testing.assert_array_equal(y.reshape(-1), [2.0, 20.0, 300.0, 3000.0])


# --------------------------------------------------------------- closed forms

@pytest.mark.parametrize("s,pb,pa", [((1, 1), (1, 2), (2, 0)), ((2, 3), (0, 3), (3, 1))])
def test_delta_kernel_is_exact_shift(s, pb, pa):
    r = rng(3)
    N, G, Cig, Cog, H, W, KH, KW = 2, 2, 3, 2, 7, 8, 4, 5
    x = r.standard_normal((N, G * Cig, H, W))
    for ci0, kh0, kw0 in [(0, 0, 0), (2, 3, 1), (1, 2, 4)]:
        w = np.zeros((G * Cog, Cig, KH, KW))
        w[:, ci0, kh0, kw0] = 1.0
        y, _ = oracle.conv2d(x, w, None, s, pb, pa, G)
        OH, OW = y.shape[2:]
        for co in range(G * Cog):
            c = (co // Cog) * Cig + ci0
            for oh in range(OH):
                for ow in range(OW):
                    ih = oh * s[0] - pb[0] + kh0
                    iw = ow * s[1] - pb[1] + kw0
                    inside = 0 <= ih < H and 0 <= iw < W
                    want = x[:, c, ih, iw] if inside else np.zeros(N)
                    assert np.array_equal(y[:, co, oh, ow], want)


def test_identity_1x1():
    x = rng(4).standard_normal((2, 5, 6, 7))
    w = np.ones((5, 1, 1, 1))
    y, _ = oracle.conv2d(x, w, None, 1, 0, 0, 5)
    assert np.array_equal(y, x)


@pytest.mark.parametrize("c", [0.5, -2.0])
def test_constant_input_closed_form(c):
    # x == c: y[co,oh,ow] = b[co] + c * sum over taps inside the input of
    # sum_ci w[co,ci,kh,kw]; an output whose window is fully inside gets
    # b + c * sum(w[co]).
    r = rng(5)
    N, G, Cig, Cog, H, W, K, s, p = 1, 3, 2, 4, 9, 9, 3, 1, 1
    x = np.full((N, G * Cig, H, W), c)
    w = np.round(r.standard_normal((G * Cog, Cig, K, K)) * 8) / 8
    b = np.round(r.standard_normal(G * Cog) * 8) / 8
    y, _ = oracle.conv2d(x, w, b, s, p, p, G)
    for co in range(G * Cog):
        full = b[co] + c * w[co].sum()
        assert y[0, co, 4, 4] == full                 # interior
        corner = b[co] + c * w[co][:, 1:, 1:].sum()  # top-left: first row/col in padding
        assert y[0, co, 0, 0] == corner
        edge = b[co] + c * w[co][:, :, 1:].sum()     # left edge: first column in padding
        assert y[0, co, 4, 0] == edge


# ------------------------------------------------------------------ shapes

@pytest.mark.parametrize("H,K,s,pb,pa", list(itertools.product(
    [1, 2, 5, 8, 56, 127], [1, 2, 3, 4, 7, 9], [1, 2, 3, 5], [0, 1, 4], [0, 2, 4])))
def test_out_size_matches_window_enumeration(H, K, s, pb, pa):
    padded = H + pb + pa
    starts = [t for t in range(-pb, H + pa) if (t + pb) % s == 0 and t + K <= H + pa]
    got = oracle.out_size(H, K, s, pb, pa)
    if padded < K:
        assert got == -1
    else:
        assert got == len(starts)
        assert got == (padded - K) // s + 1


def test_out_size_matches_torch_shapes():
    for (H, K, s, pb, pa) in [(56, 3, 2, 1, 1), (128, 9, 2, 4, 4), (112, 4, 1, 1, 2), (7, 5, 3, 0, 2)]:
        x = torch.zeros(1, 1, H, H, dtype=torch.float64)
        w = torch.zeros(1, 1, K, K, dtype=torch.float64)
        ref = F.conv2d(F.pad(x, (pb, pa, pb, pa)), w, stride=s).shape[-1]
        assert oracle.out_size(H, K, s, pb, pa) == ref


# -------------------------------------------------------------- invariants

def test_linearity():
    x1, w1, _ = random_case(11, 2, 2, 3, 2, 6, 7, 3, 4, bias=False)
    x2, w2, _ = random_case(12, 2, 2, 3, 2, 6, 7, 3, 4, bias=False)
    args = ((2, 1), (1, 2), (2, 1), 2)
    ya, _ = oracle.conv2d(2.0 * x1 - 3.0 * x2, w1, None, *args)
    yb = 2.0 * oracle.conv2d(x1, w1, None, *args)[0] - 3.0 * oracle.conv2d(x2, w1, None, *args)[0]
    np.testing.assert_allclose(ya, yb, rtol=1e-12, atol=1e-12)
    yc, _ = oracle.conv2d(x1, w1 + w2, None, *args)
    yd = oracle.conv2d(x1, w1, None, *args)[0] + oracle.conv2d(x1, w2, None, *args)[0]
    np.testing.assert_allclose(yc, yd, rtol=1e-12, atol=1e-12)


def test_stride_is_subsampling():
    x, w, b = random_case(13, 1, 3, 2, 2, 11, 13, 5, 3)
    y1, _ = oracle.conv2d(x, w, b, 1, (2, 1), (2, 1), 2)
    y23, _ = oracle.conv2d(x, w, b, (2, 3), (2, 1), (2, 1), 2)
    np.testing.assert_array_equal(y23, y1[:, :, ::2, ::3][:, :, :y23.shape[2], :y23.shape[3]])


def test_asymmetric_padding_equals_explicit_pad():
    x, w, b = random_case(14, 2, 1, 4, 3, 9, 8, 4, 4)
    y, _ = oracle.conv2d(x, w, b, (1, 2), (1, 3), (2, 0), 3)
    xp = np.pad(x, ((0, 0), (0, 0), (1, 2), (3, 0)))
    y0, _ = oracle.conv2d(xp, w, b, (1, 2), 0, 0, 3)
    np.testing.assert_array_equal(y, y0)


def test_grouped_is_concat_of_dense():
    G, Cig, Cog = 3, 4, 2
    x, w, b = random_case(15, 2, Cig, Cog, G, 7, 7, 3, 3)
    y, _ = oracle.conv2d(x, w, b, 2, 1, 1, G)
    parts = [oracle.conv2d(x[:, g * Cig:(g + 1) * Cig], w[g * Cog:(g + 1) * Cog],
                           b[g * Cog:(g + 1) * Cog], 2, 1, 1, 1)[0] for g in range(G)]
    np.testing.assert_array_equal(y, np.concatenate(parts, axis=1))


def test_multiplier_is_sliced_depthwise():
    C, m = 3, 4
    x, w, b = random_case(16, 1, 1, m, C, 8, 9, 4, 4)
    y, _ = oracle.conv2d(x, w, b, 1, 1, 2, C)
    for j in range(m):
        yj, _ = oracle.conv2d(x, w[j::m], b[j::m], 1, 1, 2, C)
        np.testing.assert_array_equal(y[:, j::m], yj)


def test_layout_independent():
    x, w, b = random_case(17, 2, 1, 1, 6, 7, 5, 3, 3)
    xt = torch.from_numpy(x).contiguous(memory_format=torch.channels_last)
    y1, _ = oracle.conv2d(x, w, b, 1, 1, 1, 6)
    y2, _ = oracle.conv2d(xt, torch.from_numpy(w), torch.from_numpy(b), 1, 1, 1, 6)
    np.testing.assert_array_equal(y1, y2)


# ---------------------------------------------------------- library check

@pytest.mark.parametrize("case", BRUTE_CASES[:6])
def test_matches_torch_cpu_float64(case):
    N, Cig, Cog, G, H, W, KH, KW, s, pb, pa = case
    x, w, b = random_case(21, N, Cig, Cog, G, H, W, KH, KW)
    y, _ = oracle.conv2d(x, w, b, s, pb, pa, G)
    xt = F.pad(torch.from_numpy(x), (pb[1], pa[1], pb[0], pa[0]))
    ref = F.conv2d(xt, torch.from_numpy(w), torch.from_numpy(b), stride=s, groups=G)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_unbatched_and_rejections():
    x = rng(22).standard_normal((2, 5, 5))
    w = rng(23).standard_normal((2, 1, 3, 3))
    y, _ = oracle.conv2d(x, w, None, 1, 1, 1, 2)
    assert y.shape == (1, 2, 5, 5)
    with pytest.raises(ValueError):
        oracle.conv2d(x, w, None, 1, 0, 0, 3)        # C_in not divisible
    with pytest.raises(ValueError):
        oracle.conv2d(x[:, :2, :2], w, None, 1, 0, 0, 2)  # window > input


def test_correct_rounding_always_passes():
    # Bias-dominated outputs: the exact value rounded to the output dtype
    # passes, through the half-ulp term; for fp16 and bf16 some of them pass
    # only through it (tol * sum|w*x| + 1e-6 alone is below the rounding
    # step there), so the term is needed and is counted.
    r = rng(31)
    x = r.standard_normal((1, 64, 6, 6)) * 1e-3
    w = r.standard_normal((64, 1, 1, 1)) * 1e-2
    b = r.uniform(-0.1, 0.1, 64)
    ref, bound = oracle.conv2d(x, w, b, 1, 0, 0, 64)
    for name, dt in (("f32", torch.float32), ("f16", torch.float16), ("bf16", torch.bfloat16)):
        rounded = torch.from_numpy(ref).to(dt)
        assert not oracle.violations(rounded, ref, bound, name).any()
        only = oracle.rounding_only(rounded, ref, bound, name)
        if name != "f32":
            assert only.any()
        # one ulp off on those elements is outside the rule
        if only.any():
            got = rounded.double().numpy().copy()
            i = tuple(np.argwhere(only)[0])
            got[i] = ref[i] + 2.5 * oracle.half_ulp(ref[i], name)
            assert oracle.violations(got, ref, bound, name)[i]


def test_half_ulp_matches_the_dtype_spacing():
    # Pinned to numpy's own float16 / float32 spacing (the gap to the next
    # representable value) on values exactly representable in each dtype,
    # including binade starts, fp16 subnormals and negative values.
    r = rng(5)
    v16 = np.concatenate([r.standard_normal(2000) * 10.0 ** r.uniform(-7, 4, 2000),
                          [1.0, 2.0, 0.5, -4.0, 2.0 ** -14, 2.0 ** -20, 65504.0]]).astype(np.float16)
    v16 = v16[np.isfinite(v16) & (v16 != 0) & (np.abs(v16) < 65504)]
    np.testing.assert_array_equal(oracle.half_ulp(v16.astype(np.float64), "f16"),
                                  np.spacing(np.abs(v16)).astype(np.float64) / 2)
    v32 = np.concatenate([r.standard_normal(2000) * 10.0 ** r.uniform(-30, 30, 2000),
                          [1.0, 2.0 ** -126, 2.0 ** -140, -8.0]]).astype(np.float32)
    np.testing.assert_array_equal(oracle.half_ulp(v32.astype(np.float64), "f32"),
                                  np.spacing(np.abs(v32)).astype(np.float64) / 2)
    # bfloat16: spacing from the bit pattern (an 8-bit significand), via torch
    vb = torch.from_numpy(r.standard_normal(2000) * 10.0 ** r.uniform(-20, 20, 2000)).to(
        torch.bfloat16)
    vb = vb[vb != 0].abs()
    nxt = (vb.view(torch.int16) + 1).view(torch.bfloat16)
    gap = nxt.double() - vb.double()
    np.testing.assert_array_equal(oracle.half_ulp(vb.double().numpy(), "bf16"),
                                  gap.numpy() / 2)
    assert oracle.half_ulp(0.0, "bf16") == 0.0
    # one rounding (fp32 -> dtype, as the kernels' output cast) never moves a
    # value by more than the term, and reaches it at midpoints
    v = r.uniform(-3, 3, 20000).astype(np.float32)
    for name, dt in (("f16", torch.float16), ("bf16", torch.bfloat16)):
        moved = np.abs(torch.from_numpy(v).to(dt).double().numpy() - v.astype(np.float64))
        ratio = moved / oracle.half_ulp(v.astype(np.float64), name)
        assert ratio.max() <= 1.0 and ratio.max() > 0.99


def test_tolerance_rule():
    ref = np.array([1.0, 1.0, 0.0])
    # fp16: tol*bound = 2e-4, + 1e-6, + half an ulp of 1.0 (2^-11 = 4.88e-4)
    bound = np.array([0.1, 0.1, 0.0])
    got = np.array([1.0 + 6.85e-4, 1.0 + 6.95e-4, 5e-7])
    assert list(oracle.violations(got, ref, bound, "f16")) == [False, True, False]
    assert oracle.violations(np.array([np.nan]), np.array([0.0]), np.array([1.0]), "f32")[0]


# ------------------------------------------------------------ golden fixtures
# tests/golden/*.txt hold tiny integer-valued cases written by
# tests/golden/make_golden.py from this oracle (the pages print no worked
# values).  They guard the oracle against silent change; the box-sum case is
# also checked against a closed form computed another way (a summed-area
# table), not by re-running the stencil.

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(path):
    fields = {}
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, _, rest = line.strip().partition(" ")
            fields[key] = rest
    ints = lambda k: tuple(int(v) for v in fields[k].split())
    arr = lambda k, shape: np.array([float(v) for v in fields[k].split()]).reshape(shape)
    return {
        "x": arr("x", ints("x_shape")), "w": arr("w", ints("w_shape")),
        "b": None if fields["b"] == "none" else np.array([float(v) for v in fields["b"].split()]),
        "y": arr("y", ints("y_shape")), "stride": ints("stride"), "pb": ints("pad_before"),
        "pa": ints("pad_after"), "groups": int(fields["groups"]), "dilation": ints("dilation"),
    }


GOLDEN_NAMES = sorted(f[:-4] for f in os.listdir(GOLDEN) if f.endswith(".txt"))


def test_golden_fixtures_exist():
    assert len(GOLDEN_NAMES) >= 4


@pytest.mark.parametrize("name", GOLDEN_NAMES)
def test_golden_fixture_reproduced(name):
    g = _read_golden(os.path.join(GOLDEN, name + ".txt"))
    y, bound = oracle.conv2d(g["x"], g["w"], g["b"], g["stride"], g["pb"], g["pa"], g["groups"],
                             g["dilation"])
    assert y.shape == g["y"].shape
    assert np.array_equal(y, g["y"])          # integer inputs: exact
    assert (bound >= np.abs(y - (0 if g["b"] is None else g["b"][None, :, None, None]))).all()


def test_golden_box_sums_match_summed_area_table():
    g = _read_golden(os.path.join(GOLDEN, "box3x3_ramp4x4.txt"))
    x = g["x"][0, 0]
    xp = np.pad(x, 1)
    S = np.zeros((xp.shape[0] + 1, xp.shape[1] + 1))
    S[1:, 1:] = xp.cumsum(0).cumsum(1)
    H, W = x.shape
    want = np.array([[S[i + 3, j + 3] - S[i, j + 3] - S[i + 3, j] + S[i, j] for j in range(W)]
                     for i in range(H)])
    assert np.array_equal(g["y"][0, 0], want)
