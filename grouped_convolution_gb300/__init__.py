"""GB300 direct-stencil depthwise / few-channel grouped convolution: 2-D and
1-D, any dilation, forward, transposed and backward.

A thin Python binding over the C ABI in ``include/gconv.h`` (``libgconv.so``,
hand-written sm_103a CUDA kernels).  This module only marshals arguments:
every step of the convolution runs in the library's kernels, and there is no
CPU fallback -- a missing library is an error.

Functions keep the ABI's names: ``conv_bind``, ``conv1d_bind``,
``conv_transpose_bind``, ``conv_transpose1d_bind``, ``out_shape_and_stride``,
``grad_input_shape_and_stride``, ``conv_dw_forward``,
``conv_grouped_forward``, ``conv_transpose_forward``,
``conv_backward_input``, ``conv_backward_weight_workspace_size``,
``conv_backward_weight``, ``conv_select_schedule``,
``conv_force_schedule``; ``conv2d``, ``conv1d``, ``conv_transpose2d``,
``conv_transpose1d`` and ``conv2d_backward`` string them together for torch
tensors.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence, Tuple

__all__ = [
    "build", "conv_bind", "out_shape_and_stride", "conv_dw_forward",
    "conv_grouped_forward", "conv_select_schedule", "conv_force_schedule",
    "conv_schedule_name", "conv_strerror", "conv_launch_count", "conv2d",
    "conv1d_bind", "conv_transpose_bind", "conv_transpose1d_bind", "conv_transpose_forward",
    "grad_input_shape_and_stride", "conv_backward_input", "conv_backward_weight_workspace_size",
    "conv_backward_weight", "conv_backward_weight_noalloc", "conv_backward_weight_noalloc_limit",
    "conv_autotune", "conv_autotune_clear", "conv_probe_fma_rate",
    "conv1d", "conv_transpose2d", "conv_transpose1d",
    "conv2d_backward", "GconvError", "SCHEDULES", "lib_path",
]

SCHEDULES = {"auto": -1, "dw_flat": 0, "dw_row8": 1, "dw_mult": 2,
             "grp_plane": 3, "grp_reduce": 4, "grp_tc": 5, "dw_line": 6, "dw_small": 7, "dw_tc": 8,
             "dw_tcl": 9}
_DTYPE_CODES = {"float32": 0, "float16": 1, "bfloat16": 2}

_lock = threading.Lock()
_lib = None


class GconvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_strerror(status)} (status {status})")


class Tensor(ctypes.Structure):
    _fields_ = [("rank", ctypes.c_int32), ("sizes", ctypes.c_int64 * 4),
                ("strides", ctypes.c_int64 * 4)]


class Desc(ctypes.Structure):
    _fields_ = [
        ("magic", ctypes.c_uint32), ("dtype", ctypes.c_int32), ("layout", ctypes.c_int32),
        ("has_bias", ctypes.c_int32), ("unbatched", ctypes.c_int32),
        ("schedule", ctypes.c_int32),
        ("N", ctypes.c_int64), ("C_in", ctypes.c_int64), ("H", ctypes.c_int64),
        ("W", ctypes.c_int64), ("C_out", ctypes.c_int64), ("groups", ctypes.c_int64),
        ("Cin_g", ctypes.c_int64), ("Cout_g", ctypes.c_int64), ("KH", ctypes.c_int64),
        ("KW", ctypes.c_int64), ("OH", ctypes.c_int64), ("OW", ctypes.c_int64),
        ("stride", ctypes.c_int32 * 2), ("pad_before", ctypes.c_int32 * 2),
        ("pad_after", ctypes.c_int32 * 2),
        ("x_strides", ctypes.c_int64 * 4), ("w_strides", ctypes.c_int64 * 4),
        ("b_stride", ctypes.c_int64), ("y_strides", ctypes.c_int64 * 4),
        ("x_dense", ctypes.c_int32), ("transposed", ctypes.c_int32),
        ("spatial_dims", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("dilation", ctypes.c_int32 * 2), ("output_padding", ctypes.c_int32 * 2),
    ]


def lib_path() -> str:
    from . import _build
    return _build.LIB


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libgconv.so for sm_103a (in-tree) and return its path."""
    from . import _build
    return _build.build(force=force, verbose=verbose)


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build the CUDA library first "
                "(grouped_convolution_gb300.build()); there is no fallback")
        lib = ctypes.CDLL(path)
        P, i32, i64, vp = ctypes.POINTER, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
        lib.conv_bind.restype = i32
        lib.conv_bind.argtypes = [P(Tensor), P(Tensor), P(Tensor), i32, P(i32), P(i32),
                                  P(i32), P(i32), i64, P(Desc)]
        lib.conv1d_bind.restype = i32
        lib.conv1d_bind.argtypes = [P(Tensor), P(Tensor), P(Tensor), i32, i32, i32, i32, i32,
                                    i64, P(Desc)]
        lib.conv_transpose_bind.restype = i32
        lib.conv_transpose_bind.argtypes = [P(Tensor), P(Tensor), P(Tensor), i32, P(i32), P(i32),
                                            P(i32), P(i32), P(i32), i64, P(Desc)]
        lib.conv_transpose1d_bind.restype = i32
        lib.conv_transpose1d_bind.argtypes = [P(Tensor), P(Tensor), P(Tensor), i32, i32, i32,
                                              i32, i32, i32, i64, P(Desc)]
        for fn in (lib.out_shape_and_stride, lib.grad_input_shape_and_stride):
            fn.restype = i32
            fn.argtypes = [P(Desc), P(i32), P(i64), P(i64)]
        for fn in (lib.conv_dw_forward, lib.conv_grouped_forward, lib.conv_transpose_forward):
            fn.restype = i32
            fn.argtypes = [P(Desc), vp, vp, vp, vp, vp]
        lib.conv_backward_input.restype = i32
        lib.conv_backward_input.argtypes = [P(Desc), vp, vp, vp, vp]
        lib.conv_backward_weight_workspace_size.restype = i32
        lib.conv_backward_weight_workspace_size.argtypes = [P(Desc), P(ctypes.c_uint64)]
        lib.conv_backward_weight.restype = i32
        lib.conv_backward_weight.argtypes = [P(Desc), vp, vp, vp, vp, vp, ctypes.c_uint64, vp]
        lib.conv_autotune.restype = i32
        lib.conv_autotune.argtypes = [P(Desc), vp, vp, vp, vp, vp, i32, P(i32),
                                      P(ctypes.c_float)]
        lib.conv_autotune_clear.restype = None
        lib.conv_autotune_clear.argtypes = []
        lib.conv_backward_weight_noalloc.restype = i32
        lib.conv_backward_weight_noalloc.argtypes = [P(Desc), vp, vp, vp, vp, vp]
        lib.conv_backward_weight_noalloc_limit.restype = ctypes.c_uint64
        lib.conv_backward_weight_noalloc_limit.argtypes = []
        lib.conv_select_schedule.restype = i32
        lib.conv_select_schedule.argtypes = [P(Desc), vp, vp, vp, vp, P(i32)]
        lib.conv_force_schedule.restype = i32
        lib.conv_force_schedule.argtypes = [i32]
        lib.conv_schedule_name.restype = ctypes.c_char_p
        lib.conv_schedule_name.argtypes = [i32]
        lib.conv_strerror.restype = ctypes.c_char_p
        lib.conv_strerror.argtypes = [i32]
        lib.conv_test_inject_launch_error.restype = None
        lib.conv_test_inject_launch_error.argtypes = [i32]
        lib.conv_last_cuda_error.restype = i32
        lib.conv_last_cuda_error.argtypes = []
        lib.conv_launch_count.restype = ctypes.c_uint64
        lib.conv_launch_count.argtypes = []
        lib.conv_version.restype = i32
        lib.conv_version.argtypes = []
        lib.conv_probe_fma_rate.restype = i32
        lib.conv_probe_fma_rate.argtypes = [i32, vp, vp, P(ctypes.c_uint64)]
        _lib = lib
        return lib


def _strerror(status: int) -> str:
    try:
        return _load().conv_strerror(status).decode()
    except Exception:  # pragma: no cover
        return "?"


def _check(status: int, what: str):
    if status != 0:
        raise GconvError(status, what)


def _pair(v, name) -> Tuple[int, int]:
    if isinstance(v, int):
        return (v, v)
    v = tuple(int(t) for t in v)
    if len(v) != 2:
        raise ValueError(f"{name} must be an int or a pair")
    return v


def geometry(sizes: Sequence[int], strides: Sequence[int]) -> Tensor:
    t = Tensor()
    t.rank = len(sizes)
    # Ranks above 4 keep their rank so the library can reject them.
    for i, (s, st) in enumerate(list(zip(sizes, strides))[:4]):
        t.sizes[i] = int(s)
        t.strides[i] = int(st)
    return t


def _dtype_code(dtype) -> int:
    name = str(dtype).replace("torch.", "")
    if name not in _DTYPE_CODES:
        raise GconvError(3, f"dtype {dtype}")
    return _DTYPE_CODES[name]


def _geo(t):
    if t is None:
        return None
    if isinstance(t, tuple):
        return geometry(*t)
    return geometry(t.shape, t.stride())


def _common_dtype(x, w, bias, dtype):
    if dtype is not None:
        return dtype
    dtype = x.dtype
    for t in (w, bias):
        if t is not None and not isinstance(t, tuple) and t.dtype != dtype:
            raise GconvError(3, "x, w and bias must share one dtype")
    return dtype


def conv_bind(x, w, bias=None, stride=1, padding_before=0, padding_after=None,
              dilation=1, groups=1, dtype=None) -> Desc:
    """Validate and canonicalise one convolution.  ``x``, ``w`` and ``bias``
    may be torch tensors or ``(sizes, strides)`` pairs (then ``dtype`` names
    the element type).  Returns the ABI's ``gconv_desc``."""
    dtype = _common_dtype(x, w, bias, dtype)
    xs, ws, bs = _geo(x), _geo(w), _geo(bias)
    arr = ctypes.c_int32 * 2
    st = arr(*_pair(stride, "stride"))
    pb = arr(*_pair(padding_before, "padding_before"))
    pa = arr(*_pair(padding_before if padding_after is None else padding_after,
                    "padding_after"))
    dl = arr(*_pair(dilation, "dilation"))
    d = Desc()
    rc = _load().conv_bind(ctypes.byref(xs), ctypes.byref(ws),
                           ctypes.byref(bs) if bs is not None else None,
                           _dtype_code(dtype), st, pb, pa, dl, int(groups), ctypes.byref(d))
    _check(rc, "conv_bind")
    return d


def conv1d_bind(x, w, bias=None, stride=1, padding_before=0, padding_after=None,
                dilation=1, groups=1, dtype=None) -> Desc:
    """1-D convolution: x [N, C, L] (or [C, L]), w [C_out, Cin_g, K]."""
    dtype = _common_dtype(x, w, bias, dtype)
    xs, ws, bs = _geo(x), _geo(w), _geo(bias)
    pa = padding_before if padding_after is None else padding_after
    d = Desc()
    rc = _load().conv1d_bind(ctypes.byref(xs), ctypes.byref(ws),
                             ctypes.byref(bs) if bs is not None else None, _dtype_code(dtype),
                             int(stride), int(padding_before), int(pa), int(dilation),
                             int(groups), ctypes.byref(d))
    _check(rc, "conv1d_bind")
    return d


def conv_transpose_bind(x, w, bias=None, stride=1, padding_before=0, padding_after=None,
                        output_padding=0, dilation=1, groups=1, dtype=None) -> Desc:
    """Transposed 2-D convolution: w is [C_in, C_out/groups, KH, KW]."""
    dtype = _common_dtype(x, w, bias, dtype)
    xs, ws, bs = _geo(x), _geo(w), _geo(bias)
    arr = ctypes.c_int32 * 2
    st = arr(*_pair(stride, "stride"))
    pb = arr(*_pair(padding_before, "padding_before"))
    pa = arr(*_pair(padding_before if padding_after is None else padding_after,
                    "padding_after"))
    op = arr(*_pair(output_padding, "output_padding"))
    dl = arr(*_pair(dilation, "dilation"))
    d = Desc()
    rc = _load().conv_transpose_bind(ctypes.byref(xs), ctypes.byref(ws),
                                     ctypes.byref(bs) if bs is not None else None,
                                     _dtype_code(dtype), st, pb, pa, op, dl, int(groups),
                                     ctypes.byref(d))
    _check(rc, "conv_transpose_bind")
    return d


def conv_transpose1d_bind(x, w, bias=None, stride=1, padding_before=0, padding_after=None,
                          output_padding=0, dilation=1, groups=1, dtype=None) -> Desc:
    """Transposed 1-D convolution: x [N, C_in, L] (or [C_in, L]), w [C_in, Cog, K]."""
    dtype = _common_dtype(x, w, bias, dtype)
    xs, ws, bs = _geo(x), _geo(w), _geo(bias)
    pa = padding_before if padding_after is None else padding_after
    d = Desc()
    rc = _load().conv_transpose1d_bind(ctypes.byref(xs), ctypes.byref(ws),
                                       ctypes.byref(bs) if bs is not None else None,
                                       _dtype_code(dtype), int(stride), int(padding_before),
                                       int(pa), int(output_padding), int(dilation), int(groups),
                                       ctypes.byref(d))
    _check(rc, "conv_transpose1d_bind")
    return d


def out_shape_and_stride(desc: Desc):
    """Output (sizes, strides) in elements, as the ABI computes them."""
    rank = ctypes.c_int32()
    sizes = (ctypes.c_int64 * 4)()
    strides = (ctypes.c_int64 * 4)()
    _check(_load().out_shape_and_stride(ctypes.byref(desc), ctypes.byref(rank), sizes, strides),
           "out_shape_and_stride")
    r = rank.value
    return tuple(sizes[:r]), tuple(strides[:r])


def grad_input_shape_and_stride(desc: Desc):
    """(sizes, strides) of dx for a forward desc: x's sizes, dense in its layout."""
    rank = ctypes.c_int32()
    sizes = (ctypes.c_int64 * 4)()
    strides = (ctypes.c_int64 * 4)()
    _check(_load().grad_input_shape_and_stride(ctypes.byref(desc), ctypes.byref(rank), sizes,
                                               strides), "grad_input_shape_and_stride")
    r = rank.value
    return tuple(sizes[:r]), tuple(strides[:r])


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def conv_dw_forward(desc: Desc, x, w, bias, y, stream=None):
    """Depthwise forward into the preallocated ``y`` (device tensors or raw
    device pointers), on ``stream`` (default: torch's current stream)."""
    _check(_load().conv_dw_forward(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(bias),
                                   _ptr(y), _stream_ptr(stream)), "conv_dw_forward")


def conv_grouped_forward(desc: Desc, x, w, bias, y, stream=None):
    """Grouped forward (1..8 input channels per group) into ``y``."""
    _check(_load().conv_grouped_forward(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(bias),
                                        _ptr(y), _stream_ptr(stream)), "conv_grouped_forward")


def conv_transpose_forward(desc: Desc, x, w, bias, y, stream=None):
    """Transposed forward into ``y`` (desc from conv_transpose[1d]_bind)."""
    _check(_load().conv_transpose_forward(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(bias),
                                          _ptr(y), _stream_ptr(stream)), "conv_transpose_forward")


def conv_backward_input(desc: Desc, gy, w, dx, stream=None):
    """dx for the forward desc, into the preallocated ``dx``."""
    _check(_load().conv_backward_input(ctypes.byref(desc), _ptr(gy), _ptr(w), _ptr(dx),
                                       _stream_ptr(stream)), "conv_backward_input")


def conv_backward_weight_workspace_size(desc: Desc) -> int:
    out = ctypes.c_uint64()
    _check(_load().conv_backward_weight_workspace_size(ctypes.byref(desc), ctypes.byref(out)),
           "conv_backward_weight_workspace_size")
    return int(out.value)


def conv_backward_weight(desc: Desc, x, gy, dw, db, workspace, workspace_bytes=None,
                         stream=None):
    """dw (dense [C_out, Cin_g, KH, KW]) and db (dense [C_out], or None)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(_load().conv_backward_weight(ctypes.byref(desc), _ptr(x), _ptr(gy), _ptr(dw),
                                        _ptr(db), _ptr(workspace), int(workspace_bytes),
                                        _stream_ptr(stream)), "conv_backward_weight")


def conv_backward_weight_noalloc(desc: Desc, x, gy, dw, db, stream=None):
    """conv_backward_weight with the library's fixed device scratch buffer
    instead of a caller workspace, for callers that cannot allocate device
    memory (see include/gconv.h)."""
    _check(_load().conv_backward_weight_noalloc(ctypes.byref(desc), _ptr(x), _ptr(gy),
                                                _ptr(dw), _ptr(db), _stream_ptr(stream)),
           "conv_backward_weight_noalloc")


def conv_backward_weight_noalloc_limit() -> int:
    """Bytes of the fixed scratch buffer conv_backward_weight_noalloc uses."""
    return int(_load().conv_backward_weight_noalloc_limit())


def conv_autotune(desc: Desc, x, w, bias, y, reps: int = 10, stream=None):
    """Time every schedule that takes this call and record the fastest for
    its shape; returns (schedule name, microseconds per launch)."""
    sch = ctypes.c_int32()
    us = ctypes.c_float()
    _check(_load().conv_autotune(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(bias), _ptr(y),
                                 _stream_ptr(stream), int(reps), ctypes.byref(sch),
                                 ctypes.byref(us)), "conv_autotune")
    return conv_schedule_name(sch.value), float(us.value)


def conv_autotune_clear() -> None:
    _load().conv_autotune_clear()


def conv_select_schedule(desc: Desc, x, w, bias, y) -> str:
    """Name of the schedule a forward call would run (no launch)."""
    out = ctypes.c_int32()
    _check(_load().conv_select_schedule(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(bias),
                                        _ptr(y), ctypes.byref(out)), "conv_select_schedule")
    return conv_schedule_name(out.value)


def conv_force_schedule(schedule) -> None:
    """Process-wide override: a schedule name, number, or "auto"/None."""
    if schedule is None:
        schedule = -1
    if isinstance(schedule, str):
        if schedule not in SCHEDULES:
            raise GconvError(11, f"schedule {schedule!r}")
        schedule = SCHEDULES[schedule]
    _check(_load().conv_force_schedule(int(schedule)), "conv_force_schedule")


def conv_schedule_name(schedule: int) -> str:
    return _load().conv_schedule_name(int(schedule)).decode()


def conv_strerror(status: int) -> str:
    return _strerror(status)


def conv_launch_count() -> int:
    return int(_load().conv_launch_count())


def conv_probe_fma_rate(trips: int, sink, stream=None) -> int:
    """Launch the FMA-rate probe kernel on `stream` (`sink`: a CUDA float
    tensor of at least SMs x resident blocks elements); returns its FMA
    count, for the caller to divide by the time it measures."""
    n = ctypes.c_uint64(0)
    _check(_load().conv_probe_fma_rate(int(trips), ctypes.c_void_p(sink.data_ptr()),
                                       _stream_ptr(stream), ctypes.byref(n)),
           "conv_probe_fma_rate")
    return int(n.value)


def conv_test_inject_launch_error(cuda_error: int) -> None:
    _load().conv_test_inject_launch_error(int(cuda_error))


def conv_last_cuda_error() -> int:
    return int(_load().conv_last_cuda_error())


def empty_output(desc: Desc, like):
    """Allocate y (torch) with exactly the sizes and strides the ABI gives."""
    import torch
    sizes, strides = out_shape_and_stride(desc)
    return torch.empty_strided(sizes, strides, dtype=like.dtype, device=like.device)


def conv2d(x, w, bias=None, stride=1, padding_before=0, padding_after=None, groups=1,
           schedule=None, out=None, stream=None, dilation=1):
    """Bind, allocate the output and run the forward on CUDA tensors."""
    if not (x.is_cuda and w.is_cuda and (bias is None or bias.is_cuda)):
        raise GconvError(1, "conv2d needs CUDA tensors (there is no CPU path)")
    d = conv_bind(x, w, bias, stride, padding_before, padding_after, dilation, groups)
    if schedule is not None:
        d.schedule = SCHEDULES[schedule] if isinstance(schedule, str) else int(schedule)
    y = empty_output(d, x) if out is None else out
    if d.Cin_g == 1:
        conv_dw_forward(d, x, w, bias, y, stream)
    else:
        conv_grouped_forward(d, x, w, bias, y, stream)
    return y


def _cuda_only(*ts):
    if not all(t is None or t.is_cuda for t in ts):
        raise GconvError(1, "needs CUDA tensors (there is no CPU path)")


def _forced(d, schedule):
    if schedule is not None:
        d.schedule = SCHEDULES[schedule] if isinstance(schedule, str) else int(schedule)


def conv1d(x, w, bias=None, stride=1, padding_before=0, padding_after=None, groups=1,
           dilation=1, schedule=None, out=None, stream=None):
    """1-D forward on CUDA tensors: x [N, C, L], w [C_out, Cin_g, K]."""
    _cuda_only(x, w, bias)
    d = conv1d_bind(x, w, bias, stride, padding_before, padding_after, dilation, groups)
    _forced(d, schedule)
    y = empty_output(d, x) if out is None else out
    conv_grouped_forward(d, x, w, bias, y, stream)
    return y


def conv_transpose2d(x, w, bias=None, stride=1, padding_before=0, padding_after=None,
                     output_padding=0, groups=1, dilation=1, schedule=None, out=None,
                     stream=None):
    """Transposed 2-D forward on CUDA tensors: w [C_in, C_out/groups, KH, KW]."""
    _cuda_only(x, w, bias)
    d = conv_transpose_bind(x, w, bias, stride, padding_before, padding_after, output_padding,
                            dilation, groups)
    _forced(d, schedule)
    y = empty_output(d, x) if out is None else out
    conv_transpose_forward(d, x, w, bias, y, stream)
    return y


def conv_transpose1d(x, w, bias=None, stride=1, padding_before=0, padding_after=None,
                     output_padding=0, groups=1, dilation=1, schedule=None, out=None,
                     stream=None):
    """Transposed 1-D forward on CUDA tensors: w [C_in, C_out/groups, K]."""
    _cuda_only(x, w, bias)
    d = conv_transpose1d_bind(x, w, bias, stride, padding_before, padding_after,
                              output_padding, dilation, groups)
    _forced(d, schedule)
    y = empty_output(d, x) if out is None else out
    conv_transpose_forward(d, x, w, bias, y, stream)
    return y


def conv2d_backward(x, w, gy, stride=1, padding_before=0, padding_after=None, groups=1,
                    dilation=1, need=("dx", "dw", "db"), schedule=None, stream=None):
    """Gradients of the 2-D forward for the output gradient ``gy`` (CUDA
    tensors).  Returns a dict with the requested "dx", "dw", "db"."""
    _cuda_only(x, w, gy)
    import torch
    d = conv_bind(x, w, None, stride, padding_before, padding_after, dilation, groups)
    _forced(d, schedule)
    out = {}
    if "dx" in need:
        sizes, strides = grad_input_shape_and_stride(d)
        dx = torch.empty_strided(sizes, strides, dtype=x.dtype, device=x.device)
        conv_backward_input(d, gy, w, dx, stream)
        out["dx"] = dx
    if "dw" in need or "db" in need:
        dw = torch.empty(tuple(w.shape), dtype=x.dtype, device=x.device)
        db = torch.empty(d.C_out, dtype=x.dtype, device=x.device) if "db" in need else None
        nbytes = conv_backward_weight_workspace_size(d)
        ws = torch.empty((nbytes + 15) // 16 * 4, dtype=torch.float32, device=x.device)
        conv_backward_weight(d, x, gy, dw, db, ws, nbytes, stream)
        if "dw" in need:
            out["dw"] = dw
        if db is not None:
            out["db"] = db
    return out


def bind(x, w, bias=None, stride=1, padding_before=0, padding_after=None, dilation=1,
         groups=1, transposed=False, output_padding=0, dtype=None) -> Desc:
    """Any of the four bindings, chosen by the weight's rank (3: 1-D, 4: 2-D)
    and ``transposed``.  For 1-D calls, (h, w) pairs give their w element."""
    def last(v):
        return v if isinstance(v, int) else int(tuple(v)[-1])
    w_rank = len(w[0]) if isinstance(w, tuple) else w.dim()
    if w_rank == 3:
        pa = padding_before if padding_after is None else padding_after
        if transposed:
            return conv_transpose1d_bind(x, w, bias, last(stride), last(padding_before),
                                         last(pa), last(output_padding), last(dilation),
                                         groups, dtype)
        return conv1d_bind(x, w, bias, last(stride), last(padding_before), last(pa),
                           last(dilation), groups, dtype)
    if transposed:
        return conv_transpose_bind(x, w, bias, stride, padding_before, padding_after,
                                   output_padding, dilation, groups, dtype)
    return conv_bind(x, w, bias, stride, padding_before, padding_after, dilation, groups,
                     dtype)


def run(desc: Desc, x, w, bias, y, stream=None):
    """The forward entry point that takes this desc (transposed, depthwise
    or grouped)."""
    if desc.transposed:
        conv_transpose_forward(desc, x, w, bias, y, stream)
    elif desc.Cin_g == 1:
        conv_dw_forward(desc, x, w, bias, y, stream)
    else:
        conv_grouped_forward(desc, x, w, bias, y, stream)
