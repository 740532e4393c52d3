"""GPU parity beyond 2^31 elements for the wider envelope: a causal 1-D
depthwise convolution and a transposed 1-D upsampling (dw_line, dw_flat)
and the weight / bias gradient of the 1-D layer.

Inputs are drawn on the GPU from a seeded generator (no value comes from the
library).  Outputs are sampled (ends, the middle, random points); each
sample is checked against the oracle applied to the slice of the input its
taps reach.  The weight gradient of a depthwise layer sums one channel's
pixels only, so sampled channels are checked against the oracle's
backward on that channel alone.
"""

import numpy as np
import pytest
import torch

import grouped_convolution_gb300 as gc
import oracle

pytestmark = pytest.mark.gpu

N, C, L, K = 8, 2048, 140000, 4      # N*C*L = 2.29e9 elements
DT = torch.bfloat16


def nlc(t):
    return t.permute(0, 2, 1)         # [N, L, C] storage viewed as [N, C, L]


def draw(shape_nlc, gen):
    t = torch.empty(shape_nlc, dtype=DT, device="cuda")
    for i in range(shape_nlc[0]):     # one sequence at a time keeps the fp32 draw small
        t[i] = torch.randn(shape_nlc[1:], generator=gen, device="cuda").to(DT)
    return t


def sample(n, c, lo, count, seed):
    rng = np.random.default_rng(seed)
    pts = [(0, 0, 0), (n - 1, c - 1, lo - 1), (n - 1, 0, lo - 1), (0, c - 1, 0),
           (n // 2, c // 2, lo // 2)]
    pts += [(int(rng.integers(0, n)), int(rng.integers(0, c)), int(rng.integers(0, lo)))
            for _ in range(count)]
    return pts


@pytest.fixture(scope="module")
def data():
    assert N * C * L > 2 ** 31
    gen = torch.Generator(device="cuda").manual_seed(5151)
    x = nlc(draw((N, L, C), gen))
    w = (torch.randn((C, 1, K), generator=gen, device="cuda") / K ** 0.5).to(DT)
    b = (torch.rand((C,), generator=gen, device="cuda") * 0.2 - 0.1).to(DT)
    yield x, w, b
    del x
    torch.cuda.empty_cache()


def test_causal_conv1d_beyond_int32(data):
    x, w, b = data
    pb, pa = K - 1, 0
    w_h, b_h = w.cpu(), b.cpu()
    for sched in ("dw_line", "dw_flat"):
        y = gc.conv1d(x, w, b, 1, pb, pa, C, schedule=sched)
        torch.cuda.synchronize()
        assert tuple(y.shape) == (N, C, L)
        pts = sample(N, C, L, 200, seed=1)
        got = torch.stack([y[p] for p in pts]).cpu()
        refs, bounds = [], []
        for (n, c, o) in pts:
            lo, hi = o - pb, o - pb + K            # the taps' input range
            win = torch.zeros((1, 1, K), dtype=DT)
            a, z = max(lo, 0), min(hi, L)
            win[0, 0, a - lo:z - lo] = x[n, c, a:z].cpu()
            ref, bound = oracle.conv1d(win, w_h[c:c + 1], b_h[c:c + 1], 1, 0, 0, 1)
            refs.append(float(ref.reshape(-1)[0]))
            bounds.append(float(bound.reshape(-1)[0]))
        bad = oracle.violations(got, np.array(refs), np.array(bounds), "bf16")
        assert not bad.any(), f"{sched}: {int(bad.sum())} of {len(pts)} samples outside tolerance"
        del y
        torch.cuda.empty_cache()


def test_transposed_upsampling_beyond_int32(data):
    x, w, b = data
    s, pb, pa = 2, 1, 1
    OL = (L - 1) * s + K - pb - pa
    w_h, b_h = w.cpu(), b.cpu()
    for sched in ("dw_line", "dw_flat"):
        y = gc.conv_transpose1d(x, w, b, s, pb, pa, 0, C, schedule=sched)
        torch.cuda.synchronize()
        assert tuple(y.shape) == (N, C, OL)
        pts = sample(N, C, OL, 200, seed=2)
        got = torch.stack([y[p] for p in pts]).cpu()
        refs, bounds = [], []
        for (n, c, o) in pts:
            # inputs i with i*s + k = o + pb for some tap k < K
            i_lo = max(0, -(-(o + pb - (K - 1)) // s))
            i_hi = min(L - 1, (o + pb) // s)
            xs = x[n:n + 1, c:c + 1, i_lo:i_hi + 1].cpu()
            # uncropped transposed output of the slice: position o + pb - i_lo*s
            pos = o + pb - i_lo * s
            ref, bound = oracle.conv_transpose2d_points(
                xs[:, :, None, :], w_h[c:c + 1, :, None, :], b_h[c:c + 1], (1, s), 0, 0,
                (0, K), 1, np.array([[0, 0, 0, pos]]))
            refs.append(float(ref[0]))
            bounds.append(float(bound[0]))
        bad = oracle.violations(got, np.array(refs), np.array(bounds), "bf16")
        assert not bad.any(), f"{sched}: {int(bad.sum())} of {len(pts)} samples outside tolerance"
        del y
        torch.cuda.empty_cache()


def test_weight_gradient_beyond_int32(data):
    x, w, _ = data
    pb, pa = K - 1, 0
    gen = torch.Generator(device="cuda").manual_seed(6262)
    gy = nlc(draw((N, L, C), gen))
    d = gc.conv1d_bind(x, w, None, 1, pb, pa, 1, C)
    dw = torch.empty((C, 1, K), dtype=DT, device="cuda")
    db = torch.empty((C,), dtype=DT, device="cuda")
    nbytes = gc.conv_backward_weight_workspace_size(d)
    ws = torch.empty(nbytes // 4 + 4, dtype=torch.float32, device="cuda")
    gc.conv_backward_weight(d, x, gy, dw, db, ws, nbytes)
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    chans = [0, C - 1] + [int(v) for v in rng.integers(0, C, 6)]
    for c in chans:
        xc = x[:, c:c + 1, :].cpu()
        gc_ = gy[:, c:c + 1, :].cpu()
        g = oracle.conv2d_backward(xc[:, :, None, :], w[c:c + 1, :, None, :].cpu(),
                                   gc_[:, :, None, :], 1, (0, pb), (0, pa), 1,
                                   need=("dw", "db"))
        got_w = dw[c].cpu().double().numpy().reshape(-1)
        ref_w, bnd_w = g["dw"][0].reshape(-1), g["dw"][1].reshape(-1)
        assert not oracle.violations(got_w, ref_w, bnd_w, "bf16").any(), f"dw channel {c}"
        got_b = np.array([float(db[c])])
        assert not oracle.violations(got_b, g["db"][0], g["db"][1], "bf16").any(), \
            f"db channel {c}"
    del gy
    torch.cuda.empty_cache()
