"""The C ABI from a plain C99 program (tests/c_abi/abi_host.c): the header
compiles as C with warnings as errors, the program links against the built
library and its host-only checks pass.  CPU only."""
import os
import shutil
import subprocess

import pytest

from newton_schulz_bucket_gb300 import _capi

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_against_the_library(tmp_path):
    lib = _capi.lib_path()
    if not os.path.exists(lib):
        pytest.skip("library not built")
    exe = tmp_path / "abi_host"
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(HERE, "c_abi", "abi_host.c"), "-L", libdir, "-lmuon_gb300",
           "-Wl,-rpath," + libdir, "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "passed" in r.stdout
