"""GPU parity beyond 2^31 elements: 64-bit offsets in every index path.

The tensors are too large for the oracle to compute in full, so outputs are
sampled (corners, the last element, random points) and each sample is
checked against the oracle applied to that output's receptive field: the
(Cin_g, KH, KW) input window, zero outside the image, with the output
channel's weights and bias.  Inputs are drawn on the GPU from a seeded
generator (no value comes from the library).
"""

import numpy as np
import pytest
import torch

import grouped_convolution_gb300 as gc
import oracle

pytestmark = pytest.mark.gpu

CASES = [
    # name, N, C_in, H, W, Cin_g, Cout_g, K, stride, pad, dtype, schedules
    ("dw3x3_bf16_cl", 16, 1024, 400, 400, 1, 1, 3, 1, 1, torch.bfloat16,
     ["dw_row8", "dw_flat", "dw_line"]),
    ("dw3x3_f16_nchw", 12, 1024, 420, 420, 1, 1, 3, 1, 1, torch.float16, ["dw_mult"]),
    ("grp4x8_9x9_bf16_cl", 64, 256, 384, 384, 4, 8, 9, 2, 4, torch.bfloat16, ["grp_tc"]),
]


def sample_points(n, co, oh, ow, count, seed):
    rng = np.random.default_rng(seed)
    pts = [(0, 0, 0, 0), (n - 1, co - 1, oh - 1, ow - 1), (n - 1, 0, oh - 1, 0),
           (0, co - 1, 0, ow - 1), (n // 2, co // 2, oh // 2, ow // 2)]
    pts += [tuple(int(rng.integers(0, m)) for m in (n, co, oh, ow)) for _ in range(count)]
    return pts


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_beyond_int32_elements(case):
    name, N, C, H, W, cig, cog, K, s, pad, dt, schedules = case
    G = C // cig
    Co = G * cog
    assert N * C * H * W > 2 ** 31
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev).manual_seed(4242)
    cl = "cl" in name
    x = torch.empty((N, H, W, C) if cl else (N, C, H, W), dtype=dt, device=dev)
    for i in range(N):   # one image at a time keeps the fp32 draw small
        x[i] = torch.randn(x.shape[1:], generator=gen, device=dev).to(dt)
    if cl:
        x = x.permute(0, 3, 1, 2)
    w = (torch.randn((Co, cig, K, K), generator=gen, device=dev) / (cig * K * K) ** 0.5).to(dt)
    b = (torch.rand((Co,), generator=gen, device=dev) * 0.2 - 0.1).to(dt)
    OH = (H + 2 * pad - K) // s + 1
    OW = (W + 2 * pad - K) // s + 1
    pts = sample_points(N, Co, OH, OW, 200, seed=len(name))
    w_h, b_h = w.cpu(), b.cpu()
    for sched in schedules:
        y = gc.conv2d(x, w, b, s, pad, pad, G, schedule=sched)
        torch.cuda.synchronize()
        assert tuple(y.shape) == (N, Co, OH, OW)
        got = torch.stack([y[p] for p in pts]).cpu()
        refs, bounds = [], []
        for (n, co, oh, ow) in pts:
            g = co // cog
            win = torch.zeros((1, cig, K, K), dtype=dt)
            ih0, iw0 = oh * s - pad, ow * s - pad
            r0, r1 = max(ih0, 0), min(ih0 + K, H)
            c0, c1 = max(iw0, 0), min(iw0 + K, W)
            win[0, :, r0 - ih0:r1 - ih0, c0 - iw0:c1 - iw0] = \
                x[n, g * cig:(g + 1) * cig, r0:r1, c0:c1].cpu()
            ref, bound = oracle.conv2d(win, w_h[co:co + 1], b_h[co:co + 1], 1, 0, 0, 1)
            refs.append(float(ref.reshape(-1)[0]))
            bounds.append(float(bound.reshape(-1)[0]))
        bad = oracle.violations(got, np.array(refs), np.array(bounds),
                                {torch.bfloat16: "bf16", torch.float16: "f16"}[dt])
        assert not bad.any(), f"{sched}: {int(bad.sum())} of {len(pts)} samples outside tolerance"
        del y
        torch.cuda.empty_cache()
