"""The C-ABI library loads and exports every entry point that
include/gconv.h declares (no GPU needed: nothing here launches)."""

import ctypes
import os
import re
import subprocess

import pytest

import grouped_convolution_gb300 as gc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gconv.h")


@pytest.fixture(scope="session")
def libpath():
    return gc.build()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "defined")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("conv_bind", "out_shape_and_stride", "conv_dw_forward",
                     "conv_grouped_forward", "conv_force_schedule", "conv_strerror",
                     "conv_select_schedule"):
        assert required in names


def test_library_exports_every_declared_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in gconv.h but not exported"


def test_exports_are_plain_c(libpath):
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True,
                         text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in declared_functions():
        assert name in exported   # unmangled, extern "C"


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "gconv.h"\nint main(void){gconv_desc d; (void)d;'
                   ' return conv_version() > 0 ? 0 : 1;}\n')
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I",
                        os.path.join(ROOT, "include"), "-c", str(src), "-o",
                        str(tmp_path / "t.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_version_and_names(libpath):
    gc.build()
    assert gc._load().conv_version() >= 100
    assert [gc.conv_schedule_name(i) for i in range(10)] == [
        "dw_flat", "dw_row8", "dw_mult", "grp_plane", "grp_reduce", "grp_tc", "dw_line",
        "dw_small", "dw_tc", "dw_tcl"]
    assert {gc.conv_schedule_name(i): i for i in range(10)} == {
        k: v for k, v in gc.SCHEDULES.items() if k != "auto"}
    assert gc.conv_schedule_name(-1) == "auto"
    assert gc.conv_schedule_name(99) == "unknown"
    assert gc.conv_strerror(0) == "ok"


def test_struct_layout_matches_c(tmp_path):
    """The ctypes mirror of gconv_desc / gconv_tensor has the C sizes and offsets."""
    src = tmp_path / "s.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "gconv.h"\n'
        'int main(void){printf("%zu %zu %zu %zu %zu\\n", sizeof(gconv_desc), '
        'sizeof(gconv_tensor), offsetof(gconv_desc, N), offsetof(gconv_desc, y_strides), '
        'offsetof(gconv_desc, x_dense)); return 0;}\n')
    exe = tmp_path / "s"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()
    assert [int(v) for v in got] == [
        ctypes.sizeof(gc.Desc), ctypes.sizeof(gc.Tensor), gc.Desc.N.offset,
        gc.Desc.y_strides.offset, gc.Desc.x_dense.offset]
