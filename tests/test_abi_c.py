"""The C ABI from a plain C99 program: include/fp8bs.h compiles as C with warnings as errors, the
calls link against libfp8bs.so, and argument errors come back from the host-side checks (no
device is touched, so this runs without a GPU)."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "fp8_fine_grained_23_b300")


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_c99_client_links_and_gets_host_side_errors():
    from fp8_fine_grained_23_b300 import build
    build.build()
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "abi_c_check")
        subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "abi_c_check.c"), "-o", exe,
                        "-L", PKG, "-lfp8bs", f"-Wl,-rpath,{PKG}"],
                       check=True, capture_output=True, text=True)
        run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
        assert run.returncode == 0, run.stdout + run.stderr
        assert "0 failure(s)" in run.stdout
