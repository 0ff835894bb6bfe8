"""The boundary as a C program sees it (no GPU): include/moe_mxfp4.h compiles as
C99, and a C program linked against the library gets the same workspace plan and
argument checks as the Python binding."""
import os
import shutil
import subprocess

import pytest

from conftest import ROOT

C_PROGRAM = r"""
#include <stdio.h>
#include "moe_mxfp4.h"
int main(void) {
    moe_mxfp4_plan_t pl;
    if (moe_mxfp4_get_plan(16, 7168, 256, 257, 9, &pl) != MOE_OK) return 2;
    size_t ws = moe_mxfp4_workspace_size(16, 7168, 256, 257, 9);
    if (ws != pl.workspace_bytes || ws == 0) return 3;
    /* bad shapes are rejected on the host, before any device work */
    if (moe_mxfp4_get_plan(16, 7000, 256, 257, 9, &pl) == MOE_OK) return 4;
    if (moe_mxfp4_forward(0, 0, 0, 0, 0, 0, 0, 0, 16, 7168, 256, 257, 17, 0) != MOE_ERR_INVALID_ARG)
        return 5;
    if (moe_mxfp4_pointer_kind(0) != -1) return 6;
    printf("%s|%zu|%d\n", moe_mxfp4_version(), ws, pl.tile_rows);
    return 0;
}
"""


def _cuda_include():
    for d in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        if d and os.path.exists(os.path.join(d, "include", "cuda_runtime_api.h")):
            return os.path.join(d, "include")
    pytest.skip("CUDA headers not found")


def test_header_is_c99():
    cc = shutil.which("gcc") or pytest.skip("no C compiler")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-x", "c",
                        "-I", _cuda_include(), os.path.join(ROOT, "include", "moe_mxfp4.h")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_links_and_plans(tmp_path):
    cc = shutil.which("gcc") or pytest.skip("no C compiler")
    from mixture_experts_mxfp4_gb300 import build

    lib = build.build()
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(lib)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", str(src), "-o", str(exe),
                        "-I", os.path.join(ROOT, "include"), "-I", _cuda_include(),
                        "-L", libdir, "-lmoe_mxfp4", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stderr)
    version, ws, rows = r.stdout.strip().split("|")
    assert "sm_103a" in version
    import mixture_experts_mxfp4_gb300 as moe

    assert int(ws) == moe.workspace_size(16, 7168, 256, 257, 9)
    assert int(rows) == 16
