"""The C ABI used from plain C: `c_abi_host.c` is compiled with gcc -std=c99
against include/sgl_attn.h, linked with the built library and run.  It makes
host-only calls (version, status strings, workspace sizes, validation that
fails before any launch, the radix tree), so it needs no GPU."""
import os
import shutil
import subprocess

import pytest

from radixattention_prefix_shared_gb300 import build as _build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_against_the_header_and_library(tmp_path):
    lib = _build.build()
    exe = tmp_path / "c_abi_host"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "c_abi_host.c"),
           "-o", str(exe), "-L", os.path.dirname(lib), "-lsgl_attn",
           "-Wl,-rpath," + os.path.dirname(lib)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stdout + res.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0 and run.stdout.strip() == "ok", run.stdout + run.stderr
