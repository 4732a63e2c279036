"""The public header is plain C: a C99 program (tests/c_abi/plan_check.c)
compiles against include/tp.h with warnings as errors, links libtp.so and
runs the host-only plan calls; the whole-block C example
(tests/c_abi/block_example.c) compiles and links against the header, the
library and the CUDA runtime (it runs in a GPU test)."""
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


def build_block_example(libdir, exe):
    """Compiles tests/c_abi/block_example.c (C11: the CUDA runtime header
    uses anonymous unions) against include/tp.h, libtp.so and libcudart."""
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c_abi", "block_example.c"),
           "-L", libdir, "-ltp", f"-Wl,-rpath,{libdir}", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}", "-lm", "-o", exe]
    return subprocess.run(cmd, capture_output=True, text=True, timeout=120)


@pytest.mark.skipif(shutil.which("gcc") is None or not os.path.isdir("/usr/local/cuda/include"),
                    reason="no C compiler or CUDA headers")
def test_block_example_compiles_and_links(libdir, tmp_path):
    r = build_block_example(libdir, str(tmp_path / "block_example"))
    assert r.returncode == 0, r.stderr
