"""Writes the golden fixtures beside it from the CPU fp64 oracle alone
(nothing here touches the CUDA library).  Each case is small, with
integer-valued inputs, so every output is an exact integer a reader can
check by hand against the operation's definition: the direct stencil of
executorch PR #25085 (description, second paragraph), y[n, co, oh, ow] =
b[co] + sum over ci of the group, kh, kw of w[co, ci, kh, kw] *
x[n, g*Cin_g + ci, oh*s - pb + kh*d, ow*s - pb + kw*d] (zero outside x).

Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402


def cases():
    """(name, x, w, b, stride, pad_before, pad_after, groups, dilation)."""
    ramp = np.arange(1, 17, dtype=np.float64).reshape(1, 1, 4, 4)
    yield ("box3x3_ramp4x4", ramp, np.ones((1, 1, 3, 3)), None, 1, 1, 1, 1, 1)
    # depthwise, multiplier 2: two kernels per input channel, a bias
    x2 = np.arange(2 * 5 * 5, dtype=np.float64).reshape(1, 2, 5, 5) % 7 - 3
    w2 = np.array([[[[1, 0, -1]]], [[[0, 2, 0]]], [[[-1, 1, 1]]], [[[1, 1, 1]]]],
                  dtype=np.float64)                                  # [4, 1, 1, 3]
    yield ("dw_mult2_1x3", x2, w2, np.array([1.0, -2.0, 0.0, 3.0]), 1, (0, 1), (0, 1), 2, 1)
    # grouped, 2 input channels per group, stride 2, asymmetric padding
    x3 = np.arange(4 * 6 * 6, dtype=np.float64).reshape(1, 4, 6, 6) % 5 - 2
    w3 = (np.arange(4 * 2 * 3 * 3, dtype=np.float64).reshape(4, 2, 3, 3) % 3) - 1
    yield ("grouped2_s2_3x3", x3, w3, None, 2, (1, 0), (0, 1), 2, 1)
    # dilation 2
    x4 = np.arange(1 * 1 * 7 * 7, dtype=np.float64).reshape(1, 1, 7, 7) % 4
    w4 = np.array([[[[1, -1], [2, 1]]]], dtype=np.float64)
    yield ("dilated2_2x2", x4, w4, None, 1, 1, 1, 1, 2)


def fmt(a):
    return " ".join(repr(float(v)) for v in np.asarray(a, dtype=np.float64).ravel())


def main():
    for name, x, w, b, s, pb, pa, g, d in cases():
        y, _ = oracle.conv2d(x, w, b, s, pb, pa, g, d)
        pb2 = pb if isinstance(pb, tuple) else (pb, pb)
        pa2 = pa if isinstance(pa, tuple) else (pa, pa)
        with open(os.path.join(HERE, name + ".txt"), "w") as f:
            f.write("# written by tests/golden/make_golden.py from the CPU fp64 oracle; the\n")
            f.write("# operation is the direct stencil of executorch PR #25085 (description,\n")
            f.write("# second paragraph); integer inputs, so every value is exact.\n")
            f.write(f"stride {s} {s}\npad_before {pb2[0]} {pb2[1]}\npad_after {pa2[0]} {pa2[1]}\n")
            f.write(f"groups {g}\ndilation {d} {d}\n")
            f.write("x_shape " + " ".join(map(str, x.shape)) + "\nx " + fmt(x) + "\n")
            f.write("w_shape " + " ".join(map(str, w.shape)) + "\nw " + fmt(w) + "\n")
            f.write("b " + ("none" if b is None else fmt(b)) + "\n")
            f.write("y_shape " + " ".join(map(str, y.shape)) + "\ny " + fmt(y) + "\n")


if __name__ == "__main__":
    main()
