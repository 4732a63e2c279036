"""The public header is plain C: a C99 program (tests/c_abi/plan_check.c)
compiles against include/tp.h with warnings as errors, links libtp.so and
runs the host-only plan calls."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libdir():
    import __graft_entry__
    __graft_entry__.build()
    return os.path.join(ROOT, "tensor_transformer_layer_03_b300")


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_c99_program_against_the_header(libdir, tmp_path):
    exe = str(tmp_path / "plan_check")
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi", "plan_check.c"), "-L", libdir, "-ltp", f"-Wl,-rpath,{libdir}",
           "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
