"""The whole-block C example (tests/c_abi/block_example.c) on the GPU: a
plain C program that allocates with cudaMalloc, packs weights, runs a
65-token prompt, the same prompt as 64 cached tokens plus one decoded
token, and checks that the two agree (it prints "ok")."""
import os
import shutil
import subprocess

import pytest

from test_c_abi_cpu import ROOT, build_block_example

pytestmark = pytest.mark.gpu


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_block_example_runs(tmp_path):
    import __graft_entry__
    __graft_entry__.build()
    libdir = os.path.join(ROOT, "tensor_transformer_layer_03_b300")
    exe = str(tmp_path / "block_example")
    r = build_block_example(libdir, exe)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
