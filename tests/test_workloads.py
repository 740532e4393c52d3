"""GPU parity at the benchmark sizes.

Each benchmark workload runs at full size, in the schedule the picker gives it
(the launch the benchmark times), and every output element is compared with
the fp64 oracle (computed in full on the host cores: the largest case is
5.4e9 multiply-adds).  Reduced copies of the same workloads (fewer images,
smaller planes) are checked under every schedule that takes them.
"""

import numpy as np
import pytest
import torch

import grouped_convolution_gb300 as gc
import oracle
from grouped_convolution_gb300.inputs import WORKLOADS, make_inputs, small_variant

pytestmark = pytest.mark.gpu


def gpu_conv(wl, x, w, b, schedule=None):
    dev = torch.device("cuda")
    xd, wd = x.to(dev), w.to(dev)
    bd = b.to(dev) if b is not None else None
    d = gc.bind(xd, wd, bd, wl.stride, wl.pad_before, wl.pad_after, wl.dilation, wl.groups,
                wl.transposed, wl.output_padding)
    if schedule is not None:
        d.schedule = gc.SCHEDULES[schedule]
    y = gc.empty_output(d, xd)
    gc.run(d, xd, wd, bd, y)
    return y


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_size_workload(name):
    wl = WORKLOADS[name]
    x, w, b = make_inputs(wl)
    y = gpu_conv(wl, x, w, b)
    torch.cuda.synchronize()
    ref, bound = oracle.reference(wl, x, w, b)
    got = y.cpu()
    assert tuple(got.shape) == ref.shape
    bad = oracle.violations(got, ref, bound, wl.dtype)
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} outside tolerance"
    # the error is also small in absolute terms against the rounding unit
    err = np.abs(got.double().numpy() - ref)
    eps = {"f32": 2.0 ** -24, "f16": 2.0 ** -11, "bf16": 2.0 ** -8}[wl.dtype]
    assert float(np.max(err / (bound + np.abs(ref) + 1e-30))) < 64 * eps


@pytest.mark.parametrize("schedule", ["dw_flat", "dw_row8", "dw_mult", "grp_plane", "grp_reduce",
                                      "grp_tc", "dw_line", "dw_small", "dw_tc",
                                      "dw_tcl"])
@pytest.mark.parametrize("name", list(WORKLOADS))
def test_reduced_workload_every_schedule(name, schedule):
    wl = small_variant(WORKLOADS[name], N=2, H=min(WORKLOADS[name].H, 29),
                       W=min(WORKLOADS[name].W, 31))
    x, w, b = make_inputs(wl)
    try:
        y = gpu_conv(wl, x, w, b, schedule)
    except gc.GconvError as e:
        if e.status in (7, 11):
            pytest.skip(f"{schedule} does not take {name}")
        raise
    torch.cuda.synchronize()
    ref, bound = oracle.reference(wl, x, w, b)
    bad = oracle.violations(y.cpu(), ref, bound, wl.dtype)
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} outside tolerance"
