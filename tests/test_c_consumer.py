"""The C ABI from plain C: include/w4a16.h compiles as C99 and C++11 with every
warning an error, and a C program linked against libw4a16.so (no Python, no
CUDA headers) calls the host-only entry points and gets what the binding gets."""

import os
import shutil
import subprocess

import pytest

from w4a16_int4_weight_gb300 import build as wbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <stdio.h>
#include "w4a16.h"

int main(void) {
    size_t total = 0, s_off = 0, z_off = 0;
    int64_t ldq = 0;
    w4a16_launch_info info;
    if (w4a16_packed_layout(28672, 8192, 64, W4A16_UINT4, W4A16_BF16, &total, &s_off, &z_off, &ldq))
        return 2;
    printf("layout %zu %zu %zu %lld\n", total, s_off, z_off, (long long)ldq);
    printf("route %d %d %d\n", w4a16_route(1, 4096, 4096, 128, W4A16_UINT4B8, W4A16_BF16, 0),
           w4a16_route(2048, 4096, 4096, 128, W4A16_UINT4B8, W4A16_BF16, 0),
           w4a16_route(2048, 4096, 4096, 128, W4A16_UINT4B8, W4A16_BF16, 1));
    if (w4a16_launch_plan(8, 4096, 4096, 128, W4A16_UINT4B8, W4A16_BF16, W4A16_PATH_AUTO, 0, 152, &info))
        return 3;
    printf("plan %d %d %d %d %lld %lld\n", info.path, info.token_tile, info.k_split, info.stages,
           (long long)info.grid, (long long)info.smem_bytes);
    if (w4a16_gemm(0, 0, 0, 0, 0, 1, 4096, 4096, 7, W4A16_UINT4B8, W4A16_BF16, 0) != W4A16_ERR_INVALID_ARG)
        return 4;
    printf("error %s\n", w4a16_last_error_string());
    printf("version %d\n", w4a16_version());
    return 0;
}
"""


@pytest.fixture(scope="module")
def lib_dir():
    wbuild.build()
    return os.path.dirname(wbuild.LIB)


@pytest.mark.parametrize("std,compiler,suffix", [("c99", "gcc", ".c"), ("c++11", "g++", ".cpp")])
def test_header_compiles_cleanly(tmp_path, std, compiler, suffix):
    if not shutil.which(compiler):
        pytest.skip(f"{compiler} not available")
    src = tmp_path / f"h{suffix}"
    src.write_text(PROGRAM)
    subprocess.run([compiler, f"-std={std}", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", INCLUDE,
                    "-c", str(src), "-o", str(tmp_path / "h.o")], check=True)


def test_c_program_agrees_with_the_binding(tmp_path, lib_dir):
    if not shutil.which("gcc"):
        pytest.skip("gcc not available")
    from w4a16_int4_weight_gb300 import binding as B
    src = tmp_path / "prog.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "prog"
    subprocess.run(["gcc", "-std=c99", "-I", INCLUDE, str(src), "-L", lib_dir, "-lw4a16",
                    f"-Wl,-rpath,{lib_dir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    fields = {ln.split(" ", 1)[0]: ln.split(" ", 1)[1] for ln in out if ln}
    assert fields["layout"].split() == [str(v) for v in B.packed_layout(28672, 8192, 64, "uint4", "bf16")]
    assert fields["route"].split() == [str(B.route(1, 4096, 4096, 128, "uint4b8", "bf16")),
                                       str(B.route(2048, 4096, 4096, 128, "uint4b8", "bf16")),
                                       str(B.route(2048, 4096, 4096, 128, "uint4b8", "bf16", True))]
    p = B.launch_plan(8, 4096, 4096, 128, "uint4b8", "bf16")
    assert fields["plan"].split() == [str(B.PATHS[p["path"]]), str(p["token_tile"]), str(p["k_split"]),
                                      str(p["stages"]), str(p["grid"]), str(p["smem_bytes"])]
    assert "group size" in fields["error"]
    assert fields["version"] == str(B.version())
