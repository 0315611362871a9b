"""The C-ABI library builds, loads without a GPU and exports what include/dg.h declares;
the Python binding's ctypes structs match the C layout."""
import ctypes
import os
import re
import subprocess

import pytest

import discrete_diffusion_block_gb300 as dgp
from discrete_diffusion_block_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dg.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ctypes.CDLL(build.LIB)


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dg_\w+)\s*\(", src)))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ("dg_init_model", "dg_prefill", "dg_denoise_step", "dg_commit_canvas", "dg_generate"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (dg_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        getattr(lib, n)


def test_binding_covers_the_header():
    assert sorted(dgp.exported_symbols()) == declared_functions()


def test_last_error_is_empty_string_without_a_call(lib):
    lib.dg_last_error.restype = ctypes.c_char_p
    assert lib.dg_last_error() == b""


def test_null_arguments_fail_cleanly_without_a_gpu(lib):
    # argument validation runs on the host before any CUDA call
    L = dgp.load()
    assert L.dg_prefill(None, None, 0) == dgp.DG_EINVAL
    assert L.dg_denoise_step(None, None) == dgp.DG_EINVAL
    assert L.dg_op_canvas_attention(*([None] * 4), 0, 1, 4, 2, 64, 128, 2, 0, None, None, 0, None) == dgp.DG_EINVAL
    assert L.dg_op_moe(*([None] * 4), 1, 64, 4, 2, 64, None, None, None, None, 0, None) == dgp.DG_EINVAL
    assert "null" in L.dg_last_error().decode()


def test_workspace_queries_are_host_only(lib):
    L = dgp.load()
    assert L.dg_op_attention_workspace_bytes(0, 0, 4, 2, 64) == 0
    assert L.dg_op_attention_workspace_bytes(2048, 256, 16, 8, 128) == 0     # split-KV merged on chip
    assert L.dg_op_moe_workspace_bytes(256, 2816, 128, 8, 704) > 256 * 8 * 2816 * 4


def test_struct_layouts_match_the_header(tmp_path):
    prog = tmp_path / "layout.c"
    lines = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{HEADER}"', "int main(void) {"]
    for st in (dgp.dg_config, dgp.dg_sampler_config, dgp.dg_stats):
        name = st.__name__
        lines.append(f'printf("{name} size %zu\\n", sizeof({name}));')
        for f, _ in st._fields_:
            lines.append(f'printf("{name}.{f} %zu\\n", offsetof({name}, {f}));')
    lines += ["return 0; }"]
    prog.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-o", str(exe), str(prog)])
    got = dict(l.rsplit(" ", 1) for l in subprocess.check_output([str(exe)], text=True).splitlines())
    for st in (dgp.dg_config, dgp.dg_sampler_config, dgp.dg_stats):
        name = st.__name__
        assert int(got[f"{name} size"]) == ctypes.sizeof(st)
        for f, _ in st._fields_:
            assert int(got[f"{name}.{f}"]) == getattr(st, f).offset, (name, f)
