"""CPU fp64 oracle for grouped / depthwise convolution: forward (2-D and, as
its H = 1 case, 1-D; any dilation), transposed, and the backward (gradients
with respect to x, w and bias).

TEST INFRASTRUCTURE, not part of the product path: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  It shares no code with the CUDA library and never imports it.

The arithmetic lives in ``conv_oracle.c`` (plain loops, fp64, OpenMP over
output planes); this module compiles it with gcc and marshals arrays.  Inputs
of any dtype are widened to float64 exactly (fp16, bf16 and fp32 all embed in
fp64) and put in dense logical NCHW order before the call, so the oracle
reads both memory layouts through one plain index function.

The parity rule it serves (from the workload contract): an element passes when
|gpu - ref| <= tol * bound + 1e-6 + r(ref), with bound = sum of |w*x| over the
taps (the bias is not a term), tol = 1e-5 (fp32), 2e-3 (fp16), 1.6e-2 (bf16)
and r(ref) = half a unit in the last place of |ref| in the output dtype.  The
r term is a reading, not part of the stated formula: the output is one
round-to-nearest-even cast of an fp32 sum, and that cast alone moves the
exact result by up to half an ulp.  When the bias dominates an output, half
an ulp of |ref| can exceed tol * sum|w*x| + 1e-6 even though the value is
correctly rounded.  Nothing wider than that one rounding step is admitted,
and `rounding_only` counts the elements that pass only because of it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 1.6e-2}
ABS_TOL = 1e-6
# Significand bits (hidden bit included) and smallest normal exponent of each
# output dtype (IEEE 754 binary32 / binary16; bfloat16 = binary32's exponent
# with an 8-bit significand).
_SIG_BITS = {"f32": 24, "f16": 11, "bf16": 8}
_EMIN = {"f32": -126, "f16": -14, "bf16": -126}
# Elements that passed only through the rounding term, summed over every
# check since import (the test session reports it per test).
ROUNDING_ONLY = {"elements": 0, "checked": 0}


def build(force: bool = False) -> str:
    """Compile conv_oracle.c into a shared library (OpenMP when available)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
            "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dp = ctypes.c_int64, ctypes.POINTER(ctypes.c_double)
            lib.oracle_out_size.restype = i64
            lib.oracle_out_size.argtypes = [i64] * 6
            lib.oracle_transposed_out_size.restype = i64
            lib.oracle_transposed_out_size.argtypes = [i64] * 7
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_num_threads.argtypes = []
            lib.oracle_set_num_threads.restype = None
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            common = [dp, dp, dp] + [i64] * 16
            ip = ctypes.POINTER(ctypes.c_int64)
            lib.oracle_conv2d_f64.restype = ctypes.c_int
            lib.oracle_conv2d_f64.argtypes = common + [dp, dp]
            lib.oracle_conv2d_f64_points.restype = ctypes.c_int
            lib.oracle_conv2d_f64_points.argtypes = common + [i64, ip, dp, dp]
            tcommon = [dp, dp, dp] + [i64] * 18
            lib.oracle_conv_transpose2d_f64.restype = ctypes.c_int
            lib.oracle_conv_transpose2d_f64.argtypes = tcommon + [dp, dp]
            lib.oracle_conv_transpose2d_f64_points.restype = ctypes.c_int
            lib.oracle_conv_transpose2d_f64_points.argtypes = tcommon + [i64, ip, dp, dp]
            lib.oracle_conv2d_backward_f64.restype = ctypes.c_int
            lib.oracle_conv2d_backward_f64.argtypes = common + [dp] * 6
            _lib = lib
    return _lib


def _as_f64(a) -> np.ndarray:
    """Widen a torch tensor or array to a dense float64 numpy array in
    logical index order (exact for fp16 / bf16 / fp32)."""
    if a is None:
        return None
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu", torch.float64).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _pair(v):
    if isinstance(v, int):
        return (v, v)
    v = tuple(int(t) for t in v)
    assert len(v) == 2
    return v


def out_size(in_size: int, k: int, s: int, pb: int, pa: int, d: int = 1) -> int:
    """Output length along one spatial dim (-1 when the window never fits)."""
    return int(_load().oracle_out_size(in_size, k, s, pb, pa, d))


def transposed_out_size(in_size: int, k: int, s: int, pb: int, pa: int, op: int = 0,
                        d: int = 1) -> int:
    """Output length of a transposed convolution along one dim (-1 when
    nothing is left after the crop, or an argument is out of range)."""
    return int(_load().oracle_transposed_out_size(in_size, k, s, pb, pa, op, d))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads the oracle's loops use from now on (results do not change)."""
    _load().oracle_set_num_threads(int(n))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double)) if a is not None else None


def _prep(x, w, b, stride, pad_before, pad_after, groups, dilation=1):
    x = _as_f64(x)
    w = _as_f64(w)
    b = _as_f64(b)
    if x.ndim == 3:
        x = x[None]
    if x.ndim != 4 or w.ndim != 4:
        raise ValueError("x must be [N,C,H,W] (or [C,H,W]); w must be [Co,Cig,KH,KW]")
    sh, sw = _pair(stride)
    pbh, pbw = _pair(pad_before)
    pah, paw = _pair(pad_before if pad_after is None else pad_after)
    N, C_in, H, W = x.shape
    C_out, Cin_g, KH, KW = w.shape
    if Cin_g * groups != C_in:
        raise ValueError("C_in must equal Cin_g * groups")
    if b is not None and b.shape != (C_out,):
        raise ValueError("bias must be [C_out]")
    dh, dw = _pair(dilation)
    OH = out_size(H, KH, sh, pbh, pah, dh)
    OW = out_size(W, KW, sw, pbw, paw, dw)
    if OH < 0 or OW < 0:
        raise ValueError("window larger than the padded input")
    dims = (N, C_in, H, W, C_out, groups, KH, KW, sh, sw, pbh, pbw, pah, paw, dh, dw)
    return x, w, b, dims, (N, C_out, OH, OW)


def conv2d(x, w, b=None, stride=1, pad_before=0, pad_after=None, groups=1, dilation=1):
    """Reference convolution.  Returns (y, bound) as float64 arrays of shape
    [N, C_out, OH, OW]."""
    x, w, b, dims, oshape = _prep(x, w, b, stride, pad_before, pad_after, groups, dilation)
    y = np.empty(oshape, dtype=np.float64)
    bound = np.empty(oshape, dtype=np.float64)
    rc = _load().oracle_conv2d_f64(_ptr(x), _ptr(w), _ptr(b), *dims, _ptr(y), _ptr(bound))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return y, bound


def conv2d_points(x, w, b, stride, pad_before, pad_after, groups, pts, dilation=1):
    """Reference values at selected outputs.  ``pts`` is an [P, 4] integer
    array of (n, co, oh, ow).  Returns (y, bound), each of length P."""
    x, w, b, dims, _ = _prep(x, w, b, stride, pad_before, pad_after, groups, dilation)
    pts = np.ascontiguousarray(np.asarray(pts, dtype=np.int64).reshape(-1, 4))
    y = np.empty(len(pts), dtype=np.float64)
    bound = np.empty(len(pts), dtype=np.float64)
    rc = _load().oracle_conv2d_f64_points(
        _ptr(x), _ptr(w), _ptr(b), *dims, len(pts),
        pts.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _ptr(y), _ptr(bound))
    if rc != 0:
        raise ValueError("oracle rejected the arguments or a point")
    return y, bound


def _prep_transposed(x, w, b, stride, pad_before, pad_after, output_padding, groups,
                     dilation):
    x = _as_f64(x)
    w = _as_f64(w)
    b = _as_f64(b)
    if x.ndim == 3:
        x = x[None]
    if x.ndim != 4 or w.ndim != 4:
        raise ValueError("x must be [N,C,H,W] (or [C,H,W]); w must be [C_in,Cog,KH,KW]")
    sh, sw = _pair(stride)
    pbh, pbw = _pair(pad_before)
    pah, paw = _pair(pad_before if pad_after is None else pad_after)
    oph, opw = _pair(output_padding)
    dh, dw = _pair(dilation)
    N, C_in, H, W = x.shape
    Cw, Cout_g, KH, KW = w.shape
    if Cw != C_in or C_in % groups:
        raise ValueError("w must be [C_in, C_out/groups, KH, KW]")
    C_out = Cout_g * groups
    if b is not None and b.shape != (C_out,):
        raise ValueError("bias must be [C_out]")
    OH = transposed_out_size(H, KH, sh, pbh, pah, oph, dh)
    OW = transposed_out_size(W, KW, sw, pbw, paw, opw, dw)
    if OH < 0 or OW < 0:
        raise ValueError("nothing left of the output after the crop")
    dims = (N, C_in, H, W, C_out, groups, KH, KW, sh, sw, pbh, pbw, pah, paw, oph, opw,
            dh, dw)
    return x, w, b, dims, (N, C_out, OH, OW)


def conv_transpose2d(x, w, b=None, stride=1, pad_before=0, pad_after=None,
                     output_padding=0, groups=1, dilation=1):
    """Reference transposed convolution (w is [C_in, C_out/groups, KH, KW]).
    Returns (y, bound) as float64 arrays of shape [N, C_out, OH, OW]."""
    x, w, b, dims, oshape = _prep_transposed(x, w, b, stride, pad_before, pad_after,
                                             output_padding, groups, dilation)
    y = np.empty(oshape, dtype=np.float64)
    bound = np.empty(oshape, dtype=np.float64)
    rc = _load().oracle_conv_transpose2d_f64(_ptr(x), _ptr(w), _ptr(b), *dims, _ptr(y),
                                             _ptr(bound))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return y, bound


def conv_transpose2d_points(x, w, b, stride, pad_before, pad_after, output_padding,
                            groups, pts, dilation=1):
    """Transposed-convolution reference values at the (n, co, oh, ow) rows of
    ``pts``.  Returns (y, bound), each of length P."""
    x, w, b, dims, _ = _prep_transposed(x, w, b, stride, pad_before, pad_after,
                                        output_padding, groups, dilation)
    pts = np.ascontiguousarray(np.asarray(pts, dtype=np.int64).reshape(-1, 4))
    y = np.empty(len(pts), dtype=np.float64)
    bound = np.empty(len(pts), dtype=np.float64)
    rc = _load().oracle_conv_transpose2d_f64_points(
        _ptr(x), _ptr(w), _ptr(b), *dims, len(pts),
        pts.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _ptr(y), _ptr(bound))
    if rc != 0:
        raise ValueError("oracle rejected the arguments or a point")
    return y, bound


def conv2d_backward(x, w, gy, stride=1, pad_before=0, pad_after=None, groups=1,
                    dilation=1, need=("dx", "dw", "db")):
    """Gradients of the forward convolution for the output gradient ``gy``
    ([N, C_out, OH, OW]).  Returns a dict with the requested entries among
    "dx" [N, C_in, H, W], "dw" [C_out, Cin_g, KH, KW] and "db" [C_out], each a
    (value, bound) pair of float64 arrays."""
    unbatched = _as_f64(x).ndim == 3
    x, w, _, dims, oshape = _prep(x, w, None, stride, pad_before, pad_after, groups,
                                  dilation)
    gy = _as_f64(gy)
    if unbatched and gy.ndim == 3:
        gy = gy[None]
    if gy.shape != oshape:
        raise ValueError(f"gy must be {oshape}")
    out = {}
    bufs = {}
    shapes = {"dx": x.shape, "dw": w.shape, "db": (w.shape[0],)}
    for k in ("dx", "dw", "db"):
        if k in need:
            bufs[k] = (np.empty(shapes[k]), np.empty(shapes[k]))
        else:
            bufs[k] = (None, None)
    rc = _load().oracle_conv2d_backward_f64(
        _ptr(x), _ptr(w), _ptr(gy), *dims,
        _ptr(bufs["dx"][0]), _ptr(bufs["dx"][1]), _ptr(bufs["dw"][0]),
        _ptr(bufs["dw"][1]), _ptr(bufs["db"][0]), _ptr(bufs["db"][1]))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    for k in need:
        v, bnd = bufs[k]
        if k == "dx" and unbatched:
            v, bnd = v[0], bnd[0]
        out[k] = (v, bnd)
    return out


# 1-D convolutions are the H = 1 case of the 2-D definitions: x [N, C, L]
# (or [C, L]) becomes [N, C, 1, L] and w [Co, Cig, K] becomes [Co, Cig, 1, K].

def _to_2d(x, w):
    x = _as_f64(x)
    w = _as_f64(w)
    if x.ndim == 2:
        x = x[None]
    if x.ndim != 3 or w.ndim != 3:
        raise ValueError("x must be [N,C,L] (or [C,L]); w must be rank 3")
    return x[:, :, None, :], w[:, :, None, :]


def conv1d(x, w, b=None, stride=1, pad_before=0, pad_after=None, groups=1, dilation=1):
    """1-D reference convolution.  Returns (y, bound) of shape [N, C_out, OL]."""
    x2, w2 = _to_2d(x, w)
    pa = pad_before if pad_after is None else pad_after
    y, bound = conv2d(x2, w2, b, (1, stride), (0, pad_before), (0, pa), groups,
                      (1, dilation))
    return y[:, :, 0, :], bound[:, :, 0, :]


def conv_transpose1d(x, w, b=None, stride=1, pad_before=0, pad_after=None,
                     output_padding=0, groups=1, dilation=1):
    """1-D reference transposed convolution (w [C_in, C_out/groups, K])."""
    x2, w2 = _to_2d(x, w)
    pa = pad_before if pad_after is None else pad_after
    y, bound = conv_transpose2d(x2, w2, b, (1, stride), (0, pad_before), (0, pa),
                                (0, output_padding), groups, (1, dilation))
    return y[:, :, 0, :], bound[:, :, 0, :]


def half_ulp(ref, dtype: str):
    """Half a unit in the last place of |ref| in the output dtype: the most
    that rounding the exact value to that dtype (to nearest) moves it.  For
    |ref| in the binade [2^(E-1), 2^E) the ulp is 2^(E - p) with p the
    significand bits; below the smallest normal 2^emin the spacing is fixed
    at 2^(emin - p + 1).  Zero for ref = 0."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    _, e = np.frexp(a)                       # a = m * 2^e, m in [0.5, 1)
    lead = np.maximum(e - 1, _EMIN[dtype])   # exponent of the binade's start
    out = np.ldexp(1.0, lead - _SIG_BITS[dtype])
    return np.where(a > 0, out, 0.0)


def _errors(got, ref, bound, dtype):
    got = _as_f64(got)
    ref = np.asarray(ref, dtype=np.float64)
    bound = np.asarray(bound, dtype=np.float64)
    with np.errstate(invalid="ignore"):
        err = np.abs(got - ref)
    return err, TOL[dtype] * bound + ABS_TOL, half_ulp(ref, dtype)


def violations(got, ref, bound, dtype: str):
    """Boolean mask of elements outside
    |got - ref| <= tol*bound + 1e-6 + half_ulp(ref).  Also adds the number of
    elements that pass only through the half-ulp term to ROUNDING_ONLY."""
    err, lim, r = _errors(got, ref, bound, dtype)
    with np.errstate(invalid="ignore"):
        bad = ~(err <= lim + r)
        only = (~bad) & ~(err <= lim)
    ROUNDING_ONLY["elements"] += int(only.sum())
    ROUNDING_ONLY["checked"] += int(err.size)
    return bad


def rounding_only(got, ref, bound, dtype: str):
    """Boolean mask of the elements that pass the parity rule only because of
    the half-ulp rounding term (they fail tol*bound + 1e-6 alone)."""
    err, lim, r = _errors(got, ref, bound, dtype)
    with np.errstate(invalid="ignore"):
        return (err <= lim + r) & ~(err <= lim)


def reference(wl, x, w, b=None):
    """The oracle function that a workload description names (duck-typed:
    stride, pad_before, pad_after, groups, dilation, transposed,
    output_padding, spatial_dims attributes; 1-D workloads use the second
    element of each pair).  Returns (y, bound)."""
    dil = getattr(wl, "dilation", (1, 1))
    tr = getattr(wl, "transposed", False)
    op = getattr(wl, "output_padding", (0, 0))
    if getattr(wl, "spatial_dims", 2) == 1:
        if tr:
            return conv_transpose1d(x, w, b, wl.stride[1], wl.pad_before[1], wl.pad_after[1],
                                    op[1], wl.groups, dil[1])
        return conv1d(x, w, b, wl.stride[1], wl.pad_before[1], wl.pad_after[1], wl.groups,
                      dil[1])
    if tr:
        return conv_transpose2d(x, w, b, wl.stride, wl.pad_before, wl.pad_after, op,
                                wl.groups, dil)
    return conv2d(x, w, b, wl.stride, wl.pad_before, wl.pad_after, wl.groups, dil)
