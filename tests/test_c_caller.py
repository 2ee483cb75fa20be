"""The C ABI from a plain C program: tests/c/abi_caller.c is compiled as C99
and as C++17 against include/oss.h, linked with the in-tree liboss.so and
run. It makes only the calls that return before touching a device, so this
runs without a GPU; it checks that the header is valid C and C++, that the
library links from a C caller without Python, and that the calls return
the statuses the header documents."""

import os
import shutil
import subprocess

import pytest

from pass_attention_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_caller.c")
LIBDIR = os.path.join(ROOT, "pass_attention_gb300")


@pytest.fixture(scope="module")
def built():
    build_lib.build()
    return os.path.join(LIBDIR, "liboss.so")


@pytest.mark.parametrize("lang", ["c", "c++"])
def test_c_caller_links_and_gets_the_documented_statuses(built, tmp_path, lang):
    compiler = "gcc" if lang == "c" else "g++"
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not installed")
    exe = str(tmp_path / f"abi_caller_{lang.replace('+', 'p')}")
    std = ["-std=c99"] if lang == "c" else ["-std=c++17"]
    cmd = [compiler, "-x", lang] + std + ["-Wall", "-Wextra", "-Werror", "-O1",
                                           "-I", os.path.join(ROOT, "include"), SRC,
                                           "-x", "none", "-L", LIBDIR, "-loss",
                                           f"-Wl,-rpath,{LIBDIR}", "-lm", "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    run = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "abi version: 1 (want 1)" in run.stdout
